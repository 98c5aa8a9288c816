"""GPU parity: libpsk (through its C ABI) against the fp64 oracle on identical seeded inputs.

Reduced-size workloads keep every structural feature of the five decode workloads (several
score chunks, several decode splits, ragged tail pages, shuffled physical blocks) while the
oracle still finishes in seconds.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from parity import check_output, compare_selection, score_tolerance

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import page_sparse_kv_gb300 as psk  # noqa: E402
from workloads.device import budgets as dev_budgets, from_torch, queries as dev_queries, to_torch, upload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from page_sparse_kv_gb300.build import build
    build()


def _oracle_summaries(w, i):
    keys = w.keys(i, 0, int(w.seq_lens[i]))
    return O.page_summaries(keys, int(w.seq_lens[i]), w.page_size, w.dtype)


def _check_cache_and_summaries(w, cache, seqs):
    summ = from_torch(cache.summaries, w.dtype)
    kc = from_torch(cache.k_cache, w.dtype)
    vc = None if cache.v_cache is None else from_torch(cache.v_cache, w.dtype)
    out = {}
    for i in seqs:
        n = int(w.seq_lens[i])
        P = -(-n // w.page_size)
        blocks = w.block_table[i, :P]
        kmin, kmax = _oracle_summaries(w, i)
        assert np.array_equal(summ[blocks, :, 0], kmin), f"kmin mismatch seq {i}"
        assert np.array_equal(summ[blocks, :, 1], kmax), f"kmax mismatch seq {i}"
        assert np.array_equal(O.logical_from_cache(kc, blocks, n, w.page_size), w.keys(i)), f"K cache seq {i}"
        if vc is not None:
            assert np.array_equal(O.logical_from_cache(vc, blocks, n, w.page_size), w.values(i)), f"V cache seq {i}"
        out[i] = (kmin, kmax)
    return out


def _run_and_check(w, cache, seqs, summaries, q_np, step_tag=""):
    B, H = w.B, w.H_kv
    scale = 1.0 / math.sqrt(w.D)
    q = to_torch(q_np, w.dtype).cuda()
    scores = torch.full((B, H, w.max_pages), float("nan"), device="cuda")
    sel = cache.score_select(q, dev_budgets(w), scores_out=scores)
    out = cache.sparse_decode(q, sel)
    dense = cache.dense_decode(q)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    sel_np = sel.cpu().numpy()
    sc_np = scores.cpu().numpy()
    out_np = from_torch(out.float(), "f32")
    dense_np = from_torch(dense.float(), "f32")
    near_ties = 0
    for i in seqs:
        n = int(cache.seq_lens[i].item())
        P = -(-n // w.page_size)
        kmin, kmax = summaries[i]
        s_ref = O.quest_scores(q_np[i], kmin, kmax, w.dtype, scale)
        tol = score_tolerance(q_np[i], kmin, kmax, w.dtype, scale)
        err = np.abs(sc_np[i, :, :P] - s_ref)
        assert np.all(err <= tol), f"{step_tag} seq {i}: score err {err.max():.3e} > tol"
        sel_use = []
        for h in range(H):
            ok, near, got, ref = compare_selection(sel_np[i, h], s_ref[h], int(w.budgets[i]))
            assert ok, f"{step_tag} seq {i} head {h}: selected {got[:8]}... vs oracle {ref[:8]}..."
            near_ties += near
            sel_use.append(got)
        keys = w_keys(w, i, n)
        vals = w_vals(w, i, n)
        ref_out = O.attend_pages(q_np[i], keys, vals, n, w.page_size, sel_use, w.dtype, scale)
        check_output(out_np[i], ref_out, w.dtype)
        ref_dense = O.dense_attention(q_np[i], keys, vals, n, w.page_size, w.dtype, scale)
        check_output(dense_np[i], ref_dense, w.dtype)
    return near_ties


# keys/values including appended tokens (set per test)
_APPENDED = {}


def w_keys(w, i, n):
    base = w.keys(i)
    extra = _APPENDED.get((id(w), i, "k"))
    return base if extra is None else np.concatenate([base, np.stack(extra)])[:n]


def w_vals(w, i, n):
    base = O.latent_values(w.keys(i), w.D_v) if w.latent else w.values(i)
    extra = _APPENDED.get((id(w), i, "v"))
    return base if extra is None else np.concatenate([base, np.stack(extra)])[:n]


@pytest.mark.parametrize("idx", [1, 3, 4, 5])
def test_reduced_workload_parity(idx):
    w = W.reduced(idx)
    cache = upload(w)
    seqs = list(range(w.B))
    summ = _check_cache_and_summaries(w, cache, seqs)
    _run_and_check(w, cache, seqs, summ, w.queries(), step_tag=f"w{idx}")


def test_decode_appends_parity():
    """Workload 2's pattern: prefill, then appended tokens, each followed by a full decode step."""
    w = W.reduced(2)
    cache = upload(w)
    i = 0
    _APPENDED[(id(w), i, "k")] = []
    _APPENDED[(id(w), i, "v")] = []
    n0 = int(w.seq_lens[0])
    kmin, kmax = _oracle_summaries(w, 0)
    kmin, kmax = list(kmin), list(kmax)
    try:
        for step in range(1, w.appends + 1):
            k_new, v_new = w.append_token(0, step)
            _APPENDED[(id(w), i, "k")].append(k_new)
            _APPENDED[(id(w), i, "v")].append(v_new)
            pos = n0 + step - 1
            cache.append(to_torch(k_new[None], w.dtype).cuda(), to_torch(v_new[None], w.dtype).cuda(),
                         torch.tensor([pos], dtype=torch.int32, device="cuda"),
                         torch.tensor([0, 1], dtype=torch.int32, device="cuda"), 1)
            cache.seq_lens += 1
            p = pos // w.page_size
            if p == len(kmin):
                kmin.append(k_new.copy())
                kmax.append(k_new.copy())
            else:
                kmin[p], kmax[p] = O.summary_after_append(kmin[p], kmax[p], k_new, pos, w.page_size, w.dtype)
            # the device summary of the tail page equals the incremental oracle rule
            summ = from_torch(cache.summaries, w.dtype)
            blk = w.block_table[0, p]
            assert np.array_equal(summ[blk, :, 0], kmin[p]) and np.array_equal(summ[blk, :, 1], kmax[p])
            _run_and_check(w, cache, [0], {0: (np.stack(kmin), np.stack(kmax))}, w.queries(step),
                           step_tag=f"append {step}")
        # incremental summaries equal a rebuild over all tokens
        n = n0 + w.appends
        full = np.concatenate([w.keys(0), np.stack(_APPENDED[(id(w), i, "k")])])
        lo, hi = O.page_summaries(full, n, w.page_size, w.dtype)
        assert np.array_equal(np.stack(kmin), lo) and np.array_equal(np.stack(kmax), hi)
    finally:
        _APPENDED.clear()


def _custom(seq_lens, budgets, ps=16, dtype="bf16", H_q=8, H_kv=2, D=128, n_hot=0, seed=7):
    return W.Workload("custom", seed, dtype, B=len(seq_lens), H_q=H_q, H_kv=H_kv, D=D, D_v=D, page_size=ps,
                      seq_lens=seq_lens, budgets=budgets, n_hot=n_hot, hot_rule="random", pool_slack=3)


@pytest.mark.parametrize("case", [
    dict(seq_lens=[1, 16, 17, 33], budgets=[2, 2, 2, 2]),             # P = 1, 1, 2, 3 pages
    dict(seq_lens=[100, 250, 16 * 40], budgets=[50, 2, 40]),           # b >= P, b = 2, b = P
    dict(seq_lens=[16 * 700 + 3, 5000], budgets=[700, 3]),             # many free slots, ragged tail
    dict(seq_lens=[64 * 9 + 1, 64 * 30], budgets=[4, 7], ps=64),       # page_size 64
    dict(seq_lens=[32 * 50 + 31, 32], budgets=[5, 3], ps=32),          # page_size 32
    dict(seq_lens=[48 * 37 + 20, 48 * 3 + 1, 47], budgets=[6, 3, 2], ps=48),   # page_size 48: three tiles a page
    dict(seq_lens=[16 * 20 + 9, 77], budgets=[6, 3], dtype="f32", D=64, H_q=4, H_kv=1),
    dict(seq_lens=[16 * 30 + 2, 300], budgets=[5, 4], D=64),
    dict(seq_lens=[16 * 70 + 3, 500], budgets=[9, 4], D=64, H_q=4, H_kv=1),   # 256-byte page runs
    dict(seq_lens=[16 * 45 + 8, 16 * 9], budgets=[7, 3], H_q=16, H_kv=4),      # 4 KV heads
    dict(seq_lens=[16 * 50 + 3, 16 * 9], budgets=[7, 3], H_q=8, H_kv=8),       # G = 1 (MHA)
    dict(seq_lens=[16 * 45 + 8, 300], budgets=[6, 4], H_q=16, H_kv=8),         # G = 2
    dict(seq_lens=[16 * 33 + 1, 77], budgets=[5, 3], D=64, H_q=4, H_kv=4),     # G = 1, D = 64
    dict(seq_lens=[16 * 61 + 2, 250], budgets=[8, 4], D=64, H_q=8, H_kv=4),    # G = 2, D = 64
    dict(seq_lens=[16 * 20 + 9, 77], budgets=[6, 3], dtype="f32", D=64, H_q=2, H_kv=2),   # fp32, G = 1
    dict(seq_lens=[16 * 27 + 4, 40], budgets=[5, 3], dtype="f32", H_q=1, H_kv=1),        # fp32, D = 128, G = 1
    dict(seq_lens=[16 * 40 + 7, 16 * 11], budgets=[6, 3], H_q=32, H_kv=16),    # two head groups, G = 2
    dict(seq_lens=[16 * 33 + 9, 300], budgets=[5, 4], H_q=64, H_kv=16),        # two head groups, G = 4
    dict(seq_lens=[16 * 47 + 3, 16 * 12, 90], budgets=[6, 4, 3], H_q=64, H_kv=8),   # G = 8
    dict(seq_lens=[16 * 60 + 11, 250], budgets=[9, 4], H_q=32, H_kv=4),          # G = 8, 4 KV heads
    dict(seq_lens=[16 * 41 + 1, 77], budgets=[7, 3], H_q=8, H_kv=1),             # G = 8, one KV head
    dict(seq_lens=[64 * 13 + 5, 64 * 4], budgets=[5, 3], ps=64, H_q=64, H_kv=8), # G = 8, 64-token pages
])
def test_edge_cases(case):
    w = _custom(**case)
    cache = upload(w)
    seqs = list(range(w.B))
    summ = _check_cache_and_summaries(w, cache, seqs)
    _run_and_check(w, cache, seqs, summ, w.queries(), step_tag=str(case))


def test_nan_junk_past_seq_len_is_never_read():
    w = _custom([16 * 5 + 3, 16 * 9 + 15], [3, 4])
    cache = upload(w, junk=float("nan"))
    summ = _check_cache_and_summaries(w, cache, [0, 1])
    _run_and_check(w, cache, [0, 1], summ, w.queries(), step_tag="nan junk")


def _custom_mla(seq_lens, budgets, ps=64, seed=11):
    return W.Workload("custom-mla", seed, "bf16", B=len(seq_lens), H_q=128, H_kv=1, D=576, D_v=512, page_size=ps,
                      seq_lens=seq_lens, budgets=budgets, n_hot=2, hot_rule="random", latent=True, pool_slack=3)


@pytest.mark.parametrize("case", [
    dict(seq_lens=[64 * 3 + 5, 17, 64 * 20], budgets=[2, 2, 5], ps=64),      # one-page and odd-half tails
    dict(seq_lens=[32 * 41 + 3, 32 * 7, 9], budgets=[5, 4, 2], ps=32),       # 32-token pages, odd page counts
    dict(seq_lens=[64 * 40 + 33, 64 * 9], budgets=[40, 9], ps=64),           # b >= P and b = P
])
def test_mla_edge_cases(case):
    w = _custom_mla(**case)
    cache = upload(w)
    seqs = list(range(w.B))
    summ = _check_cache_and_summaries(w, cache, seqs)
    _run_and_check(w, cache, seqs, summ, w.queries(), step_tag="mla " + str(case))


@pytest.mark.parametrize("B, budget", [(80, 3), (2, 3), (2, 7)])
def test_mla_split_counts(B, budget):
    """The latent decode's merge with one split per (sequence, half) (80 sequences: 160 units, more
    than the SMs, so each unit gets one split and merges on its own) and with clusters of 3 and 7
    splits (value-dim slices of 88 and 40 dims, the last one shorter)."""
    rng = np.random.default_rng(B * 10 + budget)
    lens = [int(x) for x in rng.integers(64 * 2, 64 * 9, size=B)]
    w = _custom_mla(lens, [budget] * B, seed=B + budget)
    cache = upload(w)
    seqs = list(range(B)) if B <= 4 else [0, 1, B // 2, B - 1]
    summ = _check_cache_and_summaries(w, cache, seqs)
    _run_and_check(w, cache, seqs, summ, w.queries(), step_tag=f"mla splits B={B} b={budget}")


@pytest.mark.parametrize("ps", [32, 64])
def test_mla_nan_junk_past_seq_len_is_never_read(ps):
    """The latent decode multiplies whole 32-row boxes: the rows past seq_len must not reach O."""
    w = _custom_mla([ps * 5 + 3, ps * 9 + ps - 1, ps * 2 + 1], [3, 4, 2], ps=ps)
    cache = upload(w, junk=float("nan"))
    summ = _check_cache_and_summaries(w, cache, [0, 1, 2])
    _run_and_check(w, cache, [0, 1, 2], summ, w.queries(), step_tag=f"mla nan junk ps {ps}")


def _qhead_tolerance(q, kmin, kmax, dtype, scale):
    """Per (query head, page) bound on fp32 accumulation error of the per-query-head score (the
    same rule as parity.score_tolerance, without the group max)."""
    qv, lo, hi = O.to_f64(q, dtype), O.to_f64(kmin, dtype), O.to_f64(kmax, dtype)
    G = qv.shape[0] // lo.shape[1]
    mag = np.maximum(np.abs(lo), np.abs(hi))
    return np.stack([np.abs(qv[g]) @ mag[:, g // G, :].T for g in range(qv.shape[0])]) * 2e-6 * scale + 1e-30


def _run_select_params(w, cache, S, W, mode, value, step_tag, per_query_head=False):
    """Score + select through the general entry (first S and last W pages kept, one budget mode,
    rows per KV head or per query head) and the sparse decode over its rows, each against the
    oracle."""
    seqs = list(range(w.B))
    summ = _check_cache_and_summaries(w, cache, seqs)
    L = cache.layout
    q_np = w.queries()
    q = to_torch(q_np, w.dtype).cuda()
    lens = [int(x) for x in w.seq_lens]
    Ps = [-(-n // w.page_size) for n in lens]
    if mode == "per_seq":
        b_seq = [int(x) for x in w.budgets]
        b_max = max(b_seq)
        kw = dict(budgets=dev_budgets(w))
    else:
        arg = dict(fraction=value) if mode == "fraction" else dict(pages=value)
        b_seq = [O.budget_for(P, sink_pages=S, window_pages=W, **arg) for P in Ps]
        b_max = O.budget_for(L.max_pages, sink_pages=S, window_pages=W, **arg)
        kw = dict(budget_fraction=value) if mode == "fraction" else dict(budget_pages=value)
    ws = psk.make_workspace(L, b_max, device="cuda")
    R = w.H_q if per_query_head else w.H_kv  # rows per sequence
    sel = torch.full((w.B, R, b_max), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((w.B, R, w.max_pages), float("nan"), device="cuda")
    psk.page_score_select_ex(L, q, cache.summaries, cache.block_table, cache.seq_lens, b_max, cache.scale, sel, ws,
                             sink_pages=S, window_pages=W, per_query_head=per_query_head, scores_out=scores, **kw)
    out = torch.empty(w.B, w.H_q, w.D_v, dtype=cache.dtype, device="cuda")
    psk.sparse_paged_decode_ex(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, sel, b_max,
                               cache.scale, out, ws, per_query_head=per_query_head)
    torch.cuda.synchronize()
    assert psk.get_device_status(ws) == 0
    sel_np, sc_np = sel.cpu().numpy(), scores.cpu().numpy()
    out_np = from_torch(out.float(), "f32")
    scale = 1.0 / math.sqrt(w.D)
    for i in seqs:
        n, P = lens[i], Ps[i]
        kmin, kmax = summ[i]
        if per_query_head:
            s_ref = O.quest_scores_per_query_head(q_np[i], kmin, kmax, w.dtype, scale)
            tol = _qhead_tolerance(q_np[i], kmin, kmax, w.dtype, scale)
        else:
            s_ref = O.quest_scores(q_np[i], kmin, kmax, w.dtype, scale)
            tol = score_tolerance(q_np[i], kmin, kmax, w.dtype, scale)
        assert np.all(np.abs(sc_np[i, :, :P] - s_ref) <= tol), f"{step_tag} seq {i}: scores"
        use = []
        for h in range(R):
            ok, near, got, ref = compare_selection(sel_np[i, h], s_ref[h], b_seq[i], S, W)
            assert ok, f"{step_tag} seq {i} head {h}: selected {got} vs oracle {ref}"
            assert len(got) == min(b_seq[i], P)
            use.append(got)
        attend = O.attend_pages_per_query_head if per_query_head else O.attend_pages
        ref_out = attend(q_np[i], w_keys(w, i, n), w_vals(w, i, n), n, w.page_size, use, w.dtype, scale)
        check_output(out_np[i], ref_out, w.dtype)


@pytest.mark.parametrize("case", [
    dict(S=1, W=1, mode="per_seq", value=None, budgets=[40, 20, 12, 3, 12]),
    dict(S=0, W=1, mode="pages", value=16, budgets=[2] * 5, dtype="f32", D=64, H_q=4, H_kv=1),
    dict(S=2, W=2, mode="fraction", value=0.05, budgets=[2] * 5, H_q=16, H_kv=8),
    dict(S=1, W=3, mode="pages", value=9, budgets=[2] * 5, D=64, H_q=32, H_kv=8),
    dict(S=1, W=1, mode="per_seq", value=None, budgets=[30, 9, 7, 3, 5], H_q=64, H_kv=8),   # G = 8
    dict(S=0, W=1, mode="pages", value=12, budgets=[2] * 5, H_q=8, H_kv=1),                # G = 8, one KV head
])
def test_per_query_head_selection(case):
    """Pages ranked and kept per query head (the EntmaxKV top-k form; S = 0 with W = 1 is its
    tail-only always-kept set); each query head attends its own pages of its KV head."""
    extra = {k: case[k] for k in ("dtype", "D", "H_q", "H_kv") if k in case}
    w = _custom([16 * 300 + 5, 16 * 77, 16 * 40 + 9, 33, 16 * 12], case["budgets"], **extra)
    cache = upload(w)
    _run_select_params(w, cache, case["S"], case["W"], case["mode"], case["value"], "per q head " + str(case),
                       per_query_head=True)


@pytest.mark.parametrize("case", [
    dict(S=4, W=8, mode="per_seq", value=None, budgets=[40, 20, 12, 3, 12]),
    dict(S=1, W=10, mode="pages", value=20, budgets=[2] * 5),
    dict(S=2, W=3, mode="fraction", value=0.05, budgets=[2] * 5),
    dict(S=3, W=2, mode="fraction", value=0.1, budgets=[2] * 5, dtype="f32", D=64, H_q=4, H_kv=1),
    dict(S=1, W=1, mode="pages", value=7, budgets=[2] * 5, H_q=64, H_kv=16),
])
def test_sink_window_and_budget_modes(case):
    """First S and last W pages always kept (inside the budget), budgets per sequence, as a fixed
    page count or as a fraction of each sequence's pages rounded by the retained-count ceiling;
    P = 301, 77, 41, 3 and 12 pages (the short ones keep every page)."""
    extra = {k: case[k] for k in ("dtype", "D", "H_q", "H_kv") if k in case}
    w = _custom([16 * 300 + 5, 16 * 77, 16 * 40 + 9, 33, 16 * 12], case["budgets"], **extra)
    cache = upload(w)
    _run_select_params(w, cache, case["S"], case["W"], case["mode"], case["value"], str(case))


@pytest.mark.parametrize("case", [
    dict(S=1, W=10, mode="pages", value=40, ps=64),    # the latent example of the configuration table, scaled
    dict(S=2, W=4, mode="fraction", value=0.05, ps=32),
])
def test_mla_sink_window_and_budget_modes(case):
    w = _custom_mla([case["ps"] * 300 + 5, case["ps"] * 90, case["ps"] * 13 + 1], [2, 2, 2], ps=case["ps"])
    cache = upload(w)
    _run_select_params(w, cache, case["S"], case["W"], case["mode"], case["value"], "mla " + str(case))


@pytest.mark.parametrize("latent", [False, True])
def test_split_score_then_select_equals_combined(latent):
    """psk_page_score followed by psk_page_select on the same workspace gives the combined call's
    scores and selected rows bit for bit."""
    if latent:
        w = _custom_mla([64 * 200 + 5, 64 * 31, 64 * 3 + 1], [20, 7, 3])
    else:
        w = _custom([16 * 700 + 3, 16 * 77, 5000, 17], [90, 9, 30, 2])
    cache = upload(w)
    L = cache.layout
    q = dev_queries(w)
    bud = dev_budgets(w)
    sc1 = torch.full((w.B, w.H_kv, w.max_pages), float("nan"), device="cuda")
    sel1 = cache.score_select(q, bud, scores_out=sc1)
    prm = psk.select_params(budgets=bud)
    sc2 = torch.full_like(sc1, float("nan"))
    sel2 = torch.full_like(sel1, -7)
    psk.page_score(L, q, cache.summaries, cache.block_table, cache.seq_lens, prm, cache.b_max, cache.scale, cache.ws,
                   scores_out=sc2)
    psk.page_select(L, cache.seq_lens, prm, cache.b_max, sel2, cache.ws)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    assert torch.equal(sel1, sel2)
    assert torch.equal(torch.nan_to_num(sc1, nan=-1e30), torch.nan_to_num(sc2, nan=-1e30))


@pytest.mark.parametrize("ps", [16, 48, 64])
def test_value_tier_in_host_memory(ps):
    """V in pinned host memory, read over NVLink-C2C (PSK_DECODE_V_HOST): the decode equals the
    device-memory decode bit for bit and the oracle; a decode append writes the new token's value
    straight into the host cache. Pages of 64 tokens are four tiles each."""
    w = _custom([ps * 75 + 5, ps * 19 + 9, ps * 40 + ps // 2 + 3, 17], [40, 9, 30, 2], ps=ps, H_q=32, H_kv=8)
    cache = upload(w)
    L = cache.layout
    q_np = w.queries()
    q = to_torch(q_np, w.dtype).cuda()
    v_host = cache.v_cache.cpu().pin_memory()
    sel = cache.score_select(q, dev_budgets(w))
    out_dev = cache.sparse_decode(q, sel)
    out_host = torch.empty_like(out_dev)
    psk.sparse_paged_decode_ex(L, q, cache.k_cache, v_host, cache.block_table, cache.seq_lens, sel, cache.b_max,
                               cache.scale, out_host, cache.ws, v_host=True)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    assert torch.equal(out_dev, out_host)
    # one decode token per sequence appended with the value written to host memory
    rng = np.random.default_rng(5)
    lens = w.seq_lens.astype(np.int64)
    k_new = W.f32_to_bf16_bits(rng.standard_normal((w.B, w.H_kv, w.D)).astype(np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((w.B, w.H_kv, w.D)).astype(np.float32))
    start = torch.from_numpy(lens.astype(np.int32)).cuda()
    cu = torch.arange(w.B + 1, dtype=torch.int32, device="cuda")
    psk.kv_append_and_summarize(L, to_torch(k_new, w.dtype).cuda(), to_torch(v_new, w.dtype).cuda(), start, cu, 1,
                                cache.k_cache, v_host, cache.summaries, cache.block_table, cache.ws)
    cache.seq_lens.copy_(torch.from_numpy((lens + 1).astype(np.int32)).cuda())
    sel2 = cache.score_select(q, dev_budgets(w))
    out2 = torch.empty_like(out_dev)
    psk.sparse_paged_decode_ex(L, q, cache.k_cache, v_host, cache.block_table, cache.seq_lens, sel2, cache.b_max,
                               cache.scale, out2, cache.ws, v_host=True)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    sel_np = sel2.cpu().numpy()
    out_np = from_torch(out2.float(), "f32")
    scale = 1.0 / math.sqrt(w.D)
    for i in range(w.B):
        n = int(lens[i]) + 1
        keys = np.concatenate([w.keys(i), k_new[i][None]])
        vals = np.concatenate([w.values(i), v_new[i][None]])
        use = [[int(x) for x in sel_np[i, h] if x >= 0] for h in range(w.H_kv)]
        check_output(out_np[i], O.attend_pages(q_np[i], keys, vals, n, w.page_size, use, w.dtype, scale), w.dtype)


def _hot_entries(sel_np, lens, ps, frac, first_slot=0):
    """(sequence, KV head, page, slot) for the first `frac` of each row's selected pages (tail pages
    included on purpose: the decode must read those from the host anyway)."""
    ents = []
    for i in range(sel_np.shape[0]):
        for h in range(sel_np.shape[1]):
            row = [int(x) for x in sel_np[i, h] if x >= 0]
            for p in row[:max(1, int(len(row) * frac))] + [row[-1]]:
                ents.append((i, h, p))
    ents = sorted(set(ents))
    return np.array([(i, h, p, first_slot + k) for k, (i, h, p) in enumerate(ents)], dtype=np.int32)


@pytest.mark.parametrize("ps", [16, 64])
def test_value_tier_hot_buffer(ps):
    """The value tier with a resident HBM hot buffer: pages with a slot are read from HBM, the rest
    (and every tail page) from pinned host memory; the output equals the device-memory decode bit
    for bit, after fills, after evictions, and with a tail page's resident copy overwritten with
    NaN. A slot index past the buffer flags PSK_DEV_BAD_SELECTED and that page is read from host."""
    w = _custom([ps * 75 + 5, ps * 19 + 9, ps * 40 + ps // 2 + 3, 17], [40, 9, 30, 2], ps=ps, H_q=32, H_kv=8)
    cache = upload(w)
    L = cache.layout
    q = dev_queries(w)
    v_host = cache.v_cache.cpu().pin_memory()
    sel = cache.score_select(q, dev_budgets(w))
    out_dev = cache.sparse_decode(q, sel)
    torch.cuda.synchronize()
    sel_np = sel.cpu().numpy()
    lens = [int(x) for x in w.seq_lens]
    ents = _hot_entries(sel_np, lens, ps, 0.6)
    n_slots = len(ents) + 3
    v_hot = torch.zeros(n_slots, ps, w.D, dtype=torch.bfloat16, device="cuda")
    v_slot = torch.full((w.B, w.H_kv, w.max_pages), -1, dtype=torch.int32, device="cuda")
    psk.value_tier_fill(L, v_host, cache.block_table, torch.from_numpy(ents).cuda(), v_hot, v_slot, cache.ws)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    vs = v_slot.cpu().numpy()
    for i, h, p, slot in ents:
        assert vs[i, h, p] == slot
        blk = w.block_table[i, p]
        assert torch.equal(v_hot[slot].cpu(), v_host[blk, :, h, :])
    assert (vs >= 0).sum() == len(ents)

    def tiered():
        out = torch.full_like(out_dev, float("nan"))
        psk.sparse_paged_decode_tiered(L, q, cache.k_cache, v_host, v_hot, v_slot, cache.block_table, cache.seq_lens,
                                       sel, cache.b_max, cache.scale, out, cache.ws)
        torch.cuda.synchronize()
        return out

    assert torch.equal(tiered(), out_dev)
    # a tail page's resident copy is never used
    Ps = [-(-n // ps) for n in lens]
    tails = [(i, h, p, slot) for i, h, p, slot in ents if p == Ps[i] - 1]
    assert tails
    for _, _, _, slot in tails:
        v_hot[slot].fill_(float("nan"))
    assert torch.equal(tiered(), out_dev)
    # evict half the entries, then run again
    ev = ents[::2].copy()
    ev[:, 3] = -1
    psk.value_tier_fill(L, v_host, cache.block_table, torch.from_numpy(ev).cuda(), v_hot, v_slot, cache.ws)
    torch.cuda.synchronize()
    assert (v_slot.cpu().numpy() >= 0).sum() == len(ents) - len(ev)
    assert torch.equal(tiered(), out_dev)
    assert psk.get_device_status(cache.ws) == 0
    # a slot past the buffer: flagged, and the page is read from the host
    i, h, p, _ = ents[1]
    v_slot[i, h, p] = n_slots + 4
    assert torch.equal(tiered(), out_dev)
    assert psk.get_device_status(cache.ws) == psk.DEV_BAD_SELECTED
    psk.clear_device_status(cache.ws)


def test_ties_resolve_to_lower_page():
    """Pages with identical keys (hence identical summaries and scores) tie; with the cutoff
    inside the tied group the lowest-indexed tied pages win."""
    w = _custom([16 * 12], [12], H_q=4, H_kv=1)
    cache = upload(w)
    keys = w.keys(0)
    src = keys[3 * 16:4 * 16].copy()
    for p in range(5, 11):   # pages 5..10 become copies of page 3 (rewritten through the append kernel)
        cache.append(to_torch(src, w.dtype).cuda(), to_torch(w.values(0)[p * 16:(p + 1) * 16], w.dtype).cuda(),
                     torch.tensor([p * 16], dtype=torch.int32, device="cuda"),
                     torch.tensor([0, 16], dtype=torch.int32, device="cuda"), 16)
        keys[p * 16:(p + 1) * 16] = src
    q = w.queries()
    kmin, kmax = O.page_summaries(keys, 16 * 12, 16, w.dtype)
    s = O.quest_scores(q[0], kmin, kmax, w.dtype, 1 / math.sqrt(w.D))[0]
    assert all(s[p] == s[3] for p in range(5, 11))
    above = sum(1 for p in (1, 2, 4) if s[p] > s[3])
    b = 2 + above + 3                                  # takes 3 of the 7 tied pages
    sel = cache.score_select(to_torch(q, w.dtype).cuda(), torch.tensor([b], dtype=torch.int32, device="cuda"))
    got = [int(x) for x in sel.cpu().numpy()[0, 0] if x >= 0]
    ref = O.select_pages(s, b)
    assert got == ref
    assert [p for p in ref if p in (3, 5, 6, 7, 8, 9, 10)] == [3, 5, 6]


def test_device_status_on_bad_block_table():
    """An out-of-range block id is caught by the kernels' own bounds checks: status bit set,
    nothing read out of bounds, no fault."""
    w = _custom([16 * 8], [3], H_q=4, H_kv=1)
    cache = upload(w)
    cache.block_table[0, 2] = w.num_blocks + 5
    q = dev_queries(w)
    sel = cache.score_select(q, dev_budgets(w))
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) & psk.DEV_BAD_BLOCK
    psk.clear_device_status(cache.ws)
    assert psk.get_device_status(cache.ws) == 0
    bad_sel = torch.tensor([[[0, 9, 3]]], dtype=torch.int32, device="cuda")  # 9 >= P = 8, not ascending
    cache.block_table[0, 2] = w.block_table[0, 2]
    cache.sparse_decode(q, bad_sel)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) & psk.DEV_BAD_SELECTED


def test_device_status_bad_budget():
    """A per-sequence budget below the always-kept count (sink + tail) or above b_max: the select
    kernel flags PSK_DEV_BAD_BUDGET and writes that sequence's rows as -1; the other sequences
    are selected normally."""
    w = _custom([16 * 20, 16 * 30 + 3, 16 * 12], [4, 4, 4], H_q=8, H_kv=2)
    cache = upload(w)
    q_np = w.queries()
    q = to_torch(q_np, w.dtype).cuda()
    for bad in (1, cache.b_max + 1):
        psk.clear_device_status(cache.ws)
        bud = torch.tensor([4, bad, 4], dtype=torch.int32, device="cuda")
        sel = cache.score_select(q, bud)
        torch.cuda.synchronize()
        assert psk.get_device_status(cache.ws) == psk.DEV_BAD_BUDGET
        sel_np = sel.cpu().numpy()
        assert np.all(sel_np[1] == -1)
        scale = 1.0 / math.sqrt(w.D)
        for i in (0, 2):
            kmin, kmax = _oracle_summaries(w, i)
            s_ref = O.quest_scores(q_np[i], kmin, kmax, w.dtype, scale)
            for h in range(w.H_kv):
                assert compare_selection(sel_np[i, h], s_ref[h], 4)[0]
    psk.clear_device_status(cache.ws)


def test_device_status_bad_seq_len():
    """seq_len 0, or more pages than a block-table row holds: score / select and decode flag
    PSK_DEV_BAD_SEQLEN, the sequence's rows are -1 and its outputs zero; the other sequences'
    outputs still match the oracle."""
    w = _custom([16 * 20, 16 * 30 + 3], [5, 5], H_q=8, H_kv=2)
    cache = upload(w)
    q_np = w.queries()
    q = to_torch(q_np, w.dtype).cuda()
    scale = 1.0 / math.sqrt(w.D)
    good_len = int(w.seq_lens[1])
    for bad_len in (0, w.max_pages * w.page_size + 1):
        psk.clear_device_status(cache.ws)
        cache.seq_lens.copy_(torch.tensor([bad_len, good_len], dtype=torch.int32, device="cuda"))
        sel = cache.score_select(q, dev_budgets(w))
        out = cache.sparse_decode(q, sel)
        dense = cache.dense_decode(q)
        torch.cuda.synchronize()
        assert psk.get_device_status(cache.ws) == psk.DEV_BAD_SEQLEN
        sel_np = sel.cpu().numpy()
        assert np.all(sel_np[0] == -1)
        assert torch.all(out[0] == 0) and torch.all(dense[0] == 0)
        kmin, kmax = _oracle_summaries(w, 1)
        s_ref = O.quest_scores(q_np[1], kmin, kmax, w.dtype, scale)
        use = []
        for h in range(w.H_kv):
            ok, _, got, _ = compare_selection(sel_np[1, h], s_ref[h], int(w.budgets[1]))
            assert ok
            use.append(got)
        ref = O.attend_pages(q_np[1], w.keys(1), w.values(1), good_len, w.page_size, use, w.dtype, scale)
        check_output(from_torch(out.float(), "f32")[1], ref, w.dtype)
        # the sparse decode checks lengths on its own too: a valid row with a bad length
        psk.clear_device_status(cache.ws)
        cache.seq_lens.copy_(torch.tensor([int(w.seq_lens[0]), good_len], dtype=torch.int32, device="cuda"))
        sel_ok = cache.score_select(q, dev_budgets(w))
        cache.seq_lens.copy_(torch.tensor([bad_len, good_len], dtype=torch.int32, device="cuda"))
        out2 = cache.sparse_decode(q, sel_ok)
        torch.cuda.synchronize()
        assert psk.get_device_status(cache.ws) == psk.DEV_BAD_SEQLEN
        assert torch.all(out2[0] == 0)
    cache.seq_lens.copy_(torch.from_numpy(w.seq_lens.astype(np.int32)).cuda())
    psk.clear_device_status(cache.ws)


def test_device_status_bad_append():
    """An append whose positions run past the block-table row, or a negative start: the append
    kernel flags PSK_DEV_BAD_APPEND and writes nothing for that page; the cache and summaries of
    every page inside the row are unchanged and still equal the oracle's."""
    w = _custom([16 * 6, 16 * 5 + 7], [3, 3], H_q=4, H_kv=1)
    cache = upload(w)
    k_before = cache.k_cache.clone()
    s_before = cache.summaries.clone()
    k_new = torch.ones(2, w.H_kv, w.D, dtype=torch.bfloat16, device="cuda")
    v_new = torch.ones(2, w.H_kv, w.D, dtype=torch.bfloat16, device="cuda")
    for start in ([w.max_pages * w.page_size, int(w.seq_lens[1])], [-3, int(w.seq_lens[1])]):
        psk.clear_device_status(cache.ws)
        # sequence 0 appends one token at the given start; sequence 1 appends nothing
        cache.append(k_new[:1], v_new[:1], torch.tensor(start, dtype=torch.int32, device="cuda"),
                     torch.tensor([0, 1, 1], dtype=torch.int32, device="cuda"), 1)
        torch.cuda.synchronize()
        assert psk.get_device_status(cache.ws) == psk.DEV_BAD_APPEND
        assert torch.equal(cache.k_cache, k_before) and torch.equal(cache.summaries, s_before)
    _check_cache_and_summaries(w, cache, [0, 1])
    psk.clear_device_status(cache.ws)


@pytest.mark.parametrize("limit", [1, 4096])
def test_device_status_bounded_wait_times_out(limit):
    """The bounded mbarrier wait every streaming kernel uses gives up on a phase that cannot
    complete (an expected transaction count with no copy issued): PSK_DEV_TIMEOUT is set, the
    kernel returns, and the context stays usable for a full step checked against the oracle."""
    w = _custom([16 * 40 + 3, 16 * 9], [6, 3], H_q=8, H_kv=2)
    cache = upload(w)
    psk.selftest_bounded_wait(cache.ws, limit)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == psk.DEV_TIMEOUT
    psk.clear_device_status(cache.ws)
    summ = _check_cache_and_summaries(w, cache, [0, 1])
    _run_and_check(w, cache, [0, 1], summ, w.queries(), step_tag="after a timed-out wait")


def test_value_tier_in_host_memory_group_of_eight():
    """The host-memory value tier with eight query heads per KV head (tensor-core tiles only):
    the decode equals the device-memory decode bit for bit, and the oracle."""
    w = _custom([16 * 75 + 5, 16 * 19 + 9, 17], [40, 9, 2], H_q=64, H_kv=8)
    cache = upload(w)
    L = cache.layout
    q_np = w.queries()
    q = to_torch(q_np, w.dtype).cuda()
    v_host = cache.v_cache.cpu().pin_memory()
    sel = cache.score_select(q, dev_budgets(w))
    out_dev = cache.sparse_decode(q, sel)
    out_host = torch.empty_like(out_dev)
    psk.sparse_paged_decode_ex(L, q, cache.k_cache, v_host, cache.block_table, cache.seq_lens, sel, cache.b_max,
                               cache.scale, out_host, cache.ws, v_host=True)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    assert torch.equal(out_dev, out_host)
    sel_np = sel.cpu().numpy()
    out_np = from_torch(out_host.float(), "f32")
    for i in range(w.B):
        n = int(w.seq_lens[i])
        use = [[int(x) for x in sel_np[i, h] if x >= 0] for h in range(w.H_kv)]
        ref = O.attend_pages(q_np[i], w.keys(i), w.values(i), n, w.page_size, use, w.dtype, cache.scale)
        check_output(out_np[i], ref, w.dtype)


def test_stream_argument_follows_torch_current_stream():
    """The binding passes torch's current stream when no stream is given (through torch's raw
    stream query): it must name the same cudaStream_t as torch.cuda.current_stream(), on the
    default stream and inside a side-stream context."""
    def raw(s):
        return s.value or 0  # ctypes gives None for a null pointer
    assert raw(psk._stream(None)) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert raw(psk._stream(None)) == side.cuda_stream != 0
    assert raw(psk._stream(None)) == torch.cuda.current_stream().cuda_stream


def test_host_argument_errors():
    w = _custom([64], [2], H_q=4, H_kv=1)
    cache = upload(w)
    q = dev_queries(w)
    with pytest.raises(psk.PskError) as e:
        psk.page_score_select(cache.layout, q, cache.summaries, cache.block_table, cache.seq_lens, dev_budgets(w),
                              w.b_max, 0.1, torch.empty(1, 1, w.b_max, dtype=torch.int32, device="cuda"),
                              cache.ws[:16])
    assert e.value.code == 3
    bad = psk.Layout(1, 6, 4, 128, 128, 16, w.num_blocks, w.max_pages)  # 6 % 4 != 0
    with pytest.raises(psk.PskError) as e:
        psk.dense_paged_decode(bad, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, 0.1,
                               torch.empty(1, 6, 128, dtype=torch.bfloat16, device="cuda"), cache.ws)
    assert e.value.code == 1


_SPLIT_CHILD = r"""
import sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import page_sparse_kv_gb300 as psk
import workloads as W
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload
w = W.Workload("custom", 7, "f32", B=3, H_q=4, H_kv=1, D=64, D_v=64, page_size=16,
               seq_lens=[16 * 300 + 5, 16 * 77, 16 * 40 + 9], budgets=[40, 23, 41], n_hot=0, hot_rule="random",
               pool_slack=3)
cache = upload(w)
q = to_torch(w.queries(), w.dtype).cuda()
sel = cache.score_select(q, dev_budgets(w))
out = cache.sparse_decode(q, sel)
torch.cuda.synchronize()
assert psk.get_device_status(cache.ws) == 0
np.save(sys.argv[2] + ".out.npy", from_torch(out.float(), "f32"))
np.save(sys.argv[2] + ".sel.npy", sel.cpu().numpy())
print("ok")
"""


def test_split_count_does_not_change_the_output(tmp_path):
    """Split-K over the page list with an LSE merge must not change the result beyond fp32
    rounding: the same sparse decode (fp32 cache) with splits of 1, 2, 7 and 64 list entries and
    the default (tapered) splits, each against the default and against the oracle. The split
    width is a tuning override read once per process, so each width runs in a child process."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs, sels = {}, {}
    for sw in (None, 1, 2, 7, 64):
        env = dict(os.environ, PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
        env.pop("PSK_DECODE_SPLIT", None)
        if sw is not None:
            env["PSK_DECODE_SPLIT"] = str(sw)
        tag = str(tmp_path / f"split{sw}")
        r = subprocess.run([sys.executable, "-c", _SPLIT_CHILD, root, tag], env=env, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
        outs[sw] = np.load(tag + ".out.npy").astype(np.float64)
        sels[sw] = np.load(tag + ".sel.npy")
    ref = outs[None]
    for sw, o in outs.items():
        assert np.array_equal(sels[sw], sels[None])
        for i in range(o.shape[0]):
            assert np.abs(o[i] - ref[i]).max() <= 1e-5 * np.abs(ref[i]).max(), f"split {sw} seq {i}"
    w = _custom([16 * 300 + 5, 16 * 77, 16 * 40 + 9], [40, 23, 41], dtype="f32", D=64, H_q=4, H_kv=1)
    q_np = w.queries()
    scale = 1.0 / math.sqrt(w.D)
    for i in range(w.B):
        n = int(w.seq_lens[i])
        use = [[int(x) for x in sels[1][i, h] if x >= 0] for h in range(w.H_kv)]
        check_output(outs[1][i], O.attend_pages(q_np[i], w.keys(i), w.values(i), n, w.page_size, use, w.dtype, scale),
                     w.dtype)


def test_full_budget_sparse_matches_dense():
    """With b >= P every page is selected; the sparse and dense calls then attend the same tokens
    (in differently sized splits, so the fp32 merge order differs) and agree to the bf16
    tolerance."""
    w = _custom([16 * 37 + 5, 16 * 64], [64, 64])
    cache = upload(w)
    q = dev_queries(w)
    sel = cache.score_select(q, dev_budgets(w))
    sp = cache.sparse_decode(q, sel)
    de = cache.dense_decode(q)
    torch.cuda.synchronize()
    check_output(from_torch(sp.float(), "f32"), from_torch(de.float(), "f32").astype(np.float64), "bf16")


_PDL_CHILD = r"""
import math, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import oracle as O
import page_sparse_kv_gb300 as psk
import workloads as W
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload
from parity import check_output
w = W.Workload("custom", 7, "bf16", B=3, H_q=8, H_kv=2, D=128, D_v=128, page_size=16,
               seq_lens=[16 * 90 + 3, 16 * 20, 500], budgets=[9, 4, 6], n_hot=0, hot_rule="random", pool_slack=3)
cache = upload(w)
q_np = w.queries()
q = to_torch(q_np, w.dtype).cuda()
sel = cache.score_select(q, dev_budgets(w))
out = cache.sparse_decode(q, sel)
torch.cuda.synchronize()
assert psk.get_device_status(cache.ws) == 0
sel_np, out_np = sel.cpu().numpy(), from_torch(out.float(), "f32")
for i in range(w.B):
    n = int(w.seq_lens[i])
    use = [[int(x) for x in sel_np[i, h] if x >= 0] for h in range(w.H_kv)]
    ref = O.attend_pages(q_np[i], w.keys(i), w.values(i), n, w.page_size, use, w.dtype, 1 / math.sqrt(w.D))
    check_output(out_np[i], ref, w.dtype)
print("ok")
"""


@pytest.mark.parametrize("mode", ["0", "2"])
def test_launch_modes_without_and_with_in_call_pdl(mode):
    """PSK_PDL=0 (plain stream order) and PSK_PDL=2 (programmatic launch only between the kernels
    of one call) give oracle-matching results; the setting is read once per process, so each runs
    in a child process."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PSK_PDL=mode, PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
    r = subprocess.run([sys.executable, "-c", _PDL_CHILD, root], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


_MLA_MERGE_CHILD = r"""
import sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import page_sparse_kv_gb300 as psk
import workloads as W
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload
for tag, w in (("reduced", W.reduced(5)),
               ("b3", W.Workload("custom-mla", 21, "bf16", B=2, H_q=128, H_kv=1, D=576, D_v=512, page_size=64,
                                 seq_lens=[64 * 6 + 17, 64 * 5], budgets=[3, 3], n_hot=2, hot_rule="random",
                                 latent=True, pool_slack=3))):
    cache = upload(w)
    q = to_torch(w.queries(), w.dtype).cuda()
    sel = cache.score_select(q, dev_budgets(w))
    out = cache.sparse_decode(q, sel)
    dense = cache.dense_decode(q)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    np.save(sys.argv[2] + "." + tag + ".out.npy", from_torch(out, w.dtype).view(np.uint16))
    np.save(sys.argv[2] + "." + tag + ".dense.npy", from_torch(dense, w.dtype).view(np.uint16))
    np.save(sys.argv[2] + "." + tag + ".sel.npy", sel.cpu().numpy())
print("ok")
"""


def test_latent_cluster_merge_equals_workspace_merge(tmp_path):
    """The latent decode merges up to 8 splits per (sequence, half) inside a thread-block cluster
    and more in the workspace, with the same arithmetic in the same order: with clusters switched
    off (PSK_MLA_CLUSTER=0, read once per process, so each form runs in a child process) the
    sparse and dense outputs must be bit-identical (clusters of 8 and of 3 splits here)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = {}
    for flag in (None, "0"):
        env = dict(os.environ, PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
        env.pop("PSK_MLA_CLUSTER", None)
        if flag is not None:
            env["PSK_MLA_CLUSTER"] = flag
        tag = str(tmp_path / f"clu{flag}")
        r = subprocess.run([sys.executable, "-c", _MLA_MERGE_CHILD, root, tag], env=env, capture_output=True,
                           text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
        res[flag] = tag
    for w in ("reduced", "b3"):
        for part in ("sel", "out", "dense"):
            a = np.load(res[None] + f".{w}.{part}.npy")
            b = np.load(res["0"] + f".{w}.{part}.npy")
            assert np.array_equal(a, b), f"{w} {part}: cluster and workspace merges differ"


_FMA_CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import test_gpu_parity as T
import workloads as W
from workloads.device import upload
cases = [W.reduced(3),
         T._custom([16 * 45 + 8, 300, 17], [6, 4, 2], H_q=16, H_kv=8),           # G = 2
         T._custom([16 * 50 + 3, 16 * 9], [7, 3], H_q=8, H_kv=8),                # G = 1
         T._custom([16 * 61 + 2, 250], [8, 4], D=64, H_q=8, H_kv=4),             # D = 64
         T._custom([16 * 70 + 3, 500], [9, 4], D=64, H_q=4, H_kv=1),             # one KV head
         T._custom([64 * 9 + 1, 64 * 30], [4, 7], ps=64)]                        # four tiles per page
for w in cases:
    cache = upload(w)
    seqs = list(range(w.B))
    summ = T._check_cache_and_summaries(w, cache, seqs)
    T._run_and_check(w, cache, seqs, summ, w.queries(), step_tag="fma " + w.name)
for extra in (dict(), dict(H_q=16, H_kv=8)):  # per-query-head rows, G = 4 and 2
    w = T._custom([16 * 300 + 5, 16 * 77, 16 * 40 + 9, 33, 16 * 12], [40, 20, 12, 3, 12], **extra)
    T._run_select_params(w, upload(w), 1, 1, "per_seq", None, "fma per q head", per_query_head=True)
print("ok")
"""


def test_fma_forms_of_the_bf16_score_and_decode():
    """bf16 caches score and decode on the tensor cores by default; PSK_SCORE_MMA=0 and
    PSK_DECODE_MMA=0 select the FMA forms of both, which must meet the same oracle checks
    (scores within the fp32 bound, selected ids, sparse and dense outputs). The settings are read
    once per process, so the FMA forms run in a child process."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PSK_SCORE_MMA="0", PSK_DECODE_MMA="0",
               PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
    r = subprocess.run([sys.executable, "-c", _FMA_CHILD, root], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


_CHUNK_CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import test_gpu_parity as T
import workloads as W
from workloads.device import upload
cases = [W.reduced(3), W.reduced(4),
         T._custom([16 * 3000 + 5, 16 * 1100 + 9, 16 * 700], [90, 40, 700], H_q=8, H_kv=2),   # 3, 2, 1 chunks; b = P
         T._custom([16 * 2100 + 3, 16 * 1025], [300, 2], D=64, H_q=4, H_kv=1)]                 # b = 2: no free slot
for w in cases:
    cache = upload(w)
    seqs = list(range(w.B))
    summ = T._check_cache_and_summaries(w, cache, seqs)
    T._run_and_check(w, cache, seqs, summ, w.queries(), step_tag="chunk 1024 " + w.name)
print("ok")
"""


def test_selection_in_small_chunks_with_merges():
    """Units longer than one selection chunk select per chunk and merge the chunk winners in the
    unit's last CTA. With PSK_SELECT_CHUNK=1024 (read once per process, so a child process) the
    reduced workloads and a few edge cases (several chunks, b = P, no free slot) take that path
    and must give the oracle's selection and outputs."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PSK_SELECT_CHUNK="1024", PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
    r = subprocess.run([sys.executable, "-c", _CHUNK_CHILD, root], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("latent", [False, True])
def test_decode_writes_into_pinned_host_output(latent):
    """The decode's output buffer may be pinned host memory (written over NVLink-C2C by the
    kernels, as the end-to-end benchmark does): the bytes equal those of a device output."""
    if latent:
        w = _custom_mla([64 * 60 + 5, 64 * 31, 64 * 3 + 1], [9, 7, 3])
    else:
        w = _custom([16 * 300 + 5, 16 * 77, 5000, 17], [40, 9, 30, 2])
    cache = upload(w)
    q = dev_queries(w)
    sel = cache.score_select(q, dev_budgets(w))
    out_dev = cache.sparse_decode(q, sel)
    out_host = torch.full(out_dev.shape, float("nan"), dtype=out_dev.dtype).pin_memory()
    cache.sparse_decode(q, sel, out=out_host)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    assert torch.equal(out_dev.cpu(), out_host)
