"""Pins of the fp64 oracle against what the method and the mathematics fix (CPU only).

Each pin checks the oracle against something other than itself: a hand-worked example,
a characterisation by brute force (box corners, subset enumeration), a library routine
(torch's scaled_dot_product_attention in float64), or an invariant the definition implies.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


def _f32(a):
    return np.asarray(a, dtype=np.float32)


# ------------------------------------------------------------------ hand-worked example
@pytest.fixture(scope="module")
def ex(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        return json.load(f)


def test_golden_summaries(ex):
    keys = _f32(ex["keys"])[:, None, :]
    kmin, kmax = O.page_summaries(keys, ex["seq_len"], ex["page_size"], "f32")
    assert np.array_equal(kmin[:, 0], _f32(ex["kmin"]))
    assert np.array_equal(kmax[:, 0], _f32(ex["kmax"]))


def test_golden_scores_and_selection(ex):
    keys = _f32(ex["keys"])[:, None, :]
    q = _f32(ex["q"])
    kmin, kmax = O.page_summaries(keys, ex["seq_len"], ex["page_size"], "f32")
    # unscaled per-query-head bounds via a one-head-per-group view
    per_head = O.quest_scores(q, np.repeat(kmin, 2, axis=1), np.repeat(kmax, 2, axis=1), "f32", 1.0)
    assert np.array_equal(per_head, np.asarray(ex["bound_per_query_head_unscaled"], dtype=np.float64))
    s = O.quest_scores(q, kmin, kmax, "f32", 1.0 / math.sqrt(ex["D"]))
    assert np.allclose(s[0] * math.sqrt(2.0), ex["score_unscaled"], rtol=0, atol=1e-15)
    for b, sel in ex["selected_by_budget"].items():
        assert O.select_pages(s[0], int(b)) == sel


def test_golden_cutoff_score(ex):
    """The cutoff (the score of the last page chosen by score), hand-derived on the worked
    example (ties included) and on a case with distinct scores."""
    s = np.asarray(ex["score_unscaled"], dtype=np.float64)
    for b, cut in ex["cutoff_by_budget_unscaled"].items():
        assert O.cutoff_score(s, int(b)) == cut, f"budget {b}"
    s = np.asarray(ex["distinct_scores_unscaled"], dtype=np.float64)
    for b, cut in ex["distinct_cutoff_by_budget"].items():
        assert O.cutoff_score(s, int(b)) == cut, f"budget {b}"


@pytest.mark.parametrize("P", [3, 5, 8, 10])
def test_cutoff_score_is_the_weakest_winner_by_enumeration(P):
    """Against subset enumeration: the cutoff is the lowest score among the pages of the unique
    winning subset (every member beats every non-member under (score desc, index asc)), and
    None exactly when no page is chosen by score. Sink / window sets of several sizes."""
    rng = np.random.default_rng(100 + P)
    for trial in range(4):
        scores = rng.integers(-3, 4, size=P).astype(np.float64) if trial < 3 else rng.standard_normal(P)
        for S, Wn in ((1, 1), (0, 1), (2, 2)):
            forced = sorted(set(range(min(S, P))) | set(range(max(0, P - Wn), P)))
            for b in range(len(forced), P + 2):
                k = min(b, P) - len(forced)
                others = [p for p in range(P) if p not in forced]
                winners = [Sub for Sub in itertools.combinations(others, k)
                           if all((scores[x], -x) > (scores[y], -y) for x in Sub for y in others if y not in Sub)]
                assert len(winners) == 1
                got = O.cutoff_score(scores, b, S, Wn)
                if k <= 0 or min(b, P) >= P:
                    assert got is None
                else:
                    assert got == min(scores[x] for x in winners[0])


def test_golden_attention(ex):
    keys = _f32(ex["keys"])[:, None, :]
    vals = _f32(ex["values"])[:, None, :]
    q = _f32(ex["q"])
    scale = 1.0 / math.sqrt(ex["D"])
    sel = ex["selected_by_budget"][str(ex["attention_budget"])]
    out = O.attend_pages(q, keys, vals, ex["seq_len"], ex["page_size"], [sel], "f32", scale)
    toks = ex["attention_tokens"]
    v = np.asarray(ex["values"], dtype=np.float64)[toks]
    for g, logits in enumerate(ex["attention_logits_unscaled"]):
        w = np.array([math.exp(scale * l) for l in logits])
        expect = (w[:, None] * v).sum(0) / w.sum()
        assert np.allclose(out[g], expect, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ S1 summaries
def _rand_keys(rng, T, H, D, dtype):
    x = rng.standard_normal((T, H, D)).astype(np.float32)
    return x if dtype == "f32" else W.f32_to_bf16_bits(x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ps,seq_len", [(16, 16 * 5 + 3), (1, 7), (4, 4), (64, 130)])
def test_summary_bounds_attained_and_tail_masked(dtype, ps, seq_len):
    rng = np.random.default_rng(ps * 1000 + seq_len)
    T = -(-seq_len // ps) * ps + ps
    keys = _rand_keys(rng, T, 3, 8, dtype)
    kmin, kmax = O.page_summaries(keys, seq_len, ps, dtype)
    v = O.to_f64(keys, dtype)
    lo, hi = O.to_f64(kmin, dtype), O.to_f64(kmax, dtype)
    for p in range(lo.shape[0]):
        page = v[p * ps:min((p + 1) * ps, seq_len)]
        assert np.all(page >= lo[p]) and np.all(page <= hi[p])
        # attained: every summary element equals the element of some token of the page
        assert np.all(np.any(page == lo[p], axis=0)) and np.all(np.any(page == hi[p], axis=0))
    # junk past seq_len changes nothing
    keys2 = keys.copy()
    keys2[seq_len:] = _rand_keys(rng, T - seq_len, 3, 8, dtype) if T > seq_len else keys2[seq_len:]
    kmin2, kmax2 = O.page_summaries(keys2, seq_len, ps, dtype)
    assert np.array_equal(kmin, kmin2) and np.array_equal(kmax, kmax2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_summary_incremental_equals_rebuild_and_order_free(dtype):
    rng = np.random.default_rng(7)
    ps, n = 16, 16 * 3 + 5
    keys = _rand_keys(rng, n, 2, 16, dtype)
    full_lo, full_hi = O.page_summaries(keys, n, ps, dtype)
    P = full_lo.shape[0]
    lo = np.zeros_like(full_lo)
    hi = np.zeros_like(full_hi)
    for t in range(n):
        p = t // ps
        lo[p], hi[p] = O.summary_after_append(lo[p], hi[p], keys[t], t, ps, dtype)
    assert np.array_equal(lo, full_lo) and np.array_equal(hi, full_hi)
    # order inside a page does not matter
    perm = np.concatenate([p * ps + rng.permutation(min(ps, n - p * ps)) for p in range(P)])
    lo2, hi2 = O.page_summaries(keys[perm], n, ps, dtype)
    assert np.array_equal(lo2, full_lo) and np.array_equal(hi2, full_hi)


def test_summary_signed_zero_order():
    # -0.0 < +0.0 in the min and max
    keys = _f32([[0.0], [-0.0]])[:, None, :]
    lo, hi = O.page_summaries(keys, 2, 2, "f32")
    assert np.signbit(lo[0, 0, 0]) and not np.signbit(hi[0, 0, 0])
    keys = _f32([[-0.0], [-0.0]])[:, None, :]
    lo, hi = O.page_summaries(keys, 2, 2, "f32")
    assert np.signbit(lo[0, 0, 0]) and np.signbit(hi[0, 0, 0])


# ------------------------------------------------------------------ S2 Quest bound
@pytest.mark.parametrize("seed", range(6))
def test_bound_equals_max_over_box_corners(seed):
    """The page bound is the maximum of the linear map x -> q.x over the axis-aligned box
    [kmin, kmax]; a linear function reaches its maximum at a corner, so enumerating all 2^D
    corners characterises the bound independently of its per-dimension formula."""
    rng = np.random.default_rng(seed)
    D, ps, P = 6, 4, 3
    keys = rng.standard_normal((P * ps, 1, D)).astype(np.float32)
    q = rng.standard_normal((1, D)).astype(np.float32)
    kmin, kmax = O.page_summaries(keys, P * ps, ps, "f32")
    s = O.quest_scores(q, kmin, kmax, "f32", 1.0)
    qd = q[0].astype(np.float64)
    for p in range(P):
        lo, hi = kmin[p, 0].astype(np.float64), kmax[p, 0].astype(np.float64)
        best = max(float(np.dot(qd, np.where(c, hi, lo))) for c in itertools.product([0, 1], repeat=D))
        assert abs(s[0, p] - best) <= 1e-12 * (1 + abs(best))


@pytest.mark.parametrize("seed", range(4))
def test_bound_dominates_every_token_logit(seed):
    rng = np.random.default_rng(100 + seed)
    H_q, H_kv, D, ps, n = 8, 2, 16, 16, 16 * 4 + 9
    keys = _rand_keys(rng, n, H_kv, D, "bf16")
    q = W.f32_to_bf16_bits(rng.standard_normal((H_q, D)).astype(np.float32))
    kmin, kmax = O.page_summaries(keys, n, ps, "bf16")
    s = O.quest_scores(q, kmin, kmax, "bf16", 1.0)
    kv, qv = O.to_f64(keys, "bf16"), O.to_f64(q, "bf16")
    G = H_q // H_kv
    for h in range(H_kv):
        for p in range(s.shape[1]):
            page = kv[p * ps:min((p + 1) * ps, n), h]
            for g in range(h * G, (h + 1) * G):
                logits = page @ qv[g]
                tol = 1e-12 * float(np.abs(qv[g]).sum() * np.abs(page).max())
                assert np.all(logits <= s[h, p] + tol)


def test_bound_is_exact_logit_at_page_size_one_and_selects_textbook_topk():
    """With one token per page the box is a point: the bound equals q.k exactly, so the
    selection equals the textbook top-k of tokens by their max-over-group logit."""
    rng = np.random.default_rng(5)
    H_q, H_kv, D, n = 4, 1, 8, 40
    keys = rng.standard_normal((n, H_kv, D)).astype(np.float32)
    q = rng.standard_normal((H_q, D)).astype(np.float32)
    kmin, kmax = O.page_summaries(keys, n, 1, "f32")
    s = O.quest_scores(q, kmin, kmax, "f32", 1.0)
    logits = torch.from_numpy(keys[:, 0].astype(np.float64)) @ torch.from_numpy(q.astype(np.float64)).T
    best = logits.max(dim=1).values
    assert torch.allclose(torch.from_numpy(s[0]), best, rtol=0, atol=1e-12)
    b = 9
    sel = O.select_pages(s[0], b)
    inner = best[1:n - 1]
    top = (torch.topk(inner, b - 2).indices + 1).tolist()
    assert sel == sorted([0, n - 1] + top)


def test_bound_group_max_and_scale():
    rng = np.random.default_rng(11)
    H_q, H_kv, D, n, ps = 8, 2, 16, 70, 16
    keys = rng.standard_normal((n, H_kv, D)).astype(np.float32)
    q = rng.standard_normal((H_q, D)).astype(np.float32)
    kmin, kmax = O.page_summaries(keys, n, ps, "f32")
    s = O.quest_scores(q, kmin, kmax, "f32", 0.25)
    G = H_q // H_kv
    for h in range(H_kv):
        singles = [O.quest_scores(q[g:g + 1], kmin[:, h:h + 1], kmax[:, h:h + 1], "f32", 1.0)[0]
                   for g in range(h * G, (h + 1) * G)]
        assert np.allclose(s[h], 0.25 * np.max(singles, axis=0), rtol=1e-15, atol=0)


def test_split_sign_identity_used_by_the_kernels():
    """sum_d max(q kmin, q kmax) == sum_d max(q,0) kmax + min(q,0) kmin  (kmin <= kmax).
    The GPU scorer evaluates the right-hand side; this guards that algebra on the CPU."""
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal((2, 1000, 32))
    lo, hi = np.minimum(a, b), np.maximum(a, b)
    q = rng.standard_normal(32)
    lhs = np.maximum(q * lo, q * hi).sum(-1)
    rhs = (np.maximum(q, 0) * hi + np.minimum(q, 0) * lo).sum(-1)
    assert np.allclose(lhs, rhs, rtol=1e-14, atol=1e-12)


# ------------------------------------------------------------------ S3 selection
@pytest.mark.parametrize("P", [1, 2, 3, 5, 8, 10])
def test_selection_brute_force_subsets(P):
    """For every budget the chosen non-forced set is the unique subset S of the right size
    in which every member beats every non-member under (score desc, index asc)."""
    rng = np.random.default_rng(P)
    for trial in range(5):
        scores = rng.integers(-3, 4, size=P).astype(np.float64)   # many ties on purpose
        if trial == 4:
            scores = np.zeros(P)
        for b in range(2, P + 2):
            sel = O.select_pages(scores, b)
            forced = [0] if P == 1 else [0, P - 1]
            k = min(b, P) - len(forced)
            others = [p for p in range(P) if p not in forced]
            winners = []
            for S in itertools.combinations(others, k):
                out = [y for y in others if y not in S]
                if all((scores[x], -x) > (scores[y], -y) for x in S for y in out):
                    winners.append(sorted(forced + list(S)))
            assert len(winners) == 1 and winners[0] == sel
            assert sel == sorted(set(sel)) and len(sel) == min(b, P)
            assert 0 in sel and (P - 1) in sel


def test_selection_tie_lower_index_wins_on_copied_page():
    rng = np.random.default_rng(21)
    ps, P, D = 16, 12, 32
    keys = rng.standard_normal((P * ps, 1, D)).astype(np.float32)
    q = rng.standard_normal((4, D)).astype(np.float32)
    kmin, kmax = O.page_summaries(keys, P * ps, ps, "f32")
    s = O.quest_scores(q, kmin, kmax, "f32", 1.0)
    X = int(np.argmax(s[0][1:P - 1])) + 1                # best non-forced page
    Y = P - 2 if X != P - 2 else 1
    lo, hi = sorted((X, Y))
    keys[hi * ps:(hi + 1) * ps] = keys[lo * ps:(lo + 1) * ps][::-1]   # identical summary
    kmin, kmax = O.page_summaries(keys, P * ps, ps, "f32")
    s = O.quest_scores(q, kmin, kmax, "f32", 1.0)
    assert s[0, lo] == s[0, hi]
    sel = O.select_pages(s[0], 3)
    assert sel == [0, lo, P - 1]
    # -0.0 and +0.0 scores tie too
    z = np.array([1.0, -0.0, 0.0, -5.0, 2.0])
    assert O.select_pages(z, 3) == [0, 1, 4]
    z = np.array([1.0, 0.0, -0.0, -5.0, 2.0])
    assert O.select_pages(z, 3) == [0, 1, 4]


def test_selection_rejects_budget_below_two():
    with pytest.raises(ValueError):
        O.select_pages(np.zeros(3), 1)
    assert O.select_pages(np.zeros(1), 1) == [0]


# ------------------------------------------------------------------ S3 always-kept sets and budget modes
SW_CASES = [(1, 1), (2, 1), (1, 3), (3, 2), (4, 4), (0, 1), (0, 3)]


@pytest.mark.parametrize("P", [1, 2, 3, 5, 7, 9])
def test_forced_set_closed_forms(P):
    """The always-kept set of sink_pages S and window_pages W is a prefix plus a suffix of the
    pages: it holds min(P, S + W) pages, all of them once S + W >= P, page 0 (when S >= 1) and
    page P - 1 always, and its complement is the contiguous run [S, P - W)."""
    assert O.forced_pages(P) == O.forced_pages(P, 1, 1) == ([0] if P == 1 else [0, P - 1])
    for S in range(1, 6):
        for W in range(1, 6):
            f = O.forced_pages(P, S, W)
            assert len(f) == min(P, S + W) and f == sorted(set(f))
            assert f[0] == 0 and f[-1] == P - 1
            rest = [p for p in range(P) if p not in f]
            assert rest == list(range(S, P - W)) if S + W < P else rest == []
    for W in range(1, 6):  # no sink: only the last W pages (the tail among them)
        f = O.forced_pages(P, 0, W)
        assert f == list(range(max(0, P - W), P)) and len(f) == min(P, W) and f[-1] == P - 1
    for bad in ((1, 0), (-1, 1)):
        with pytest.raises(ValueError):
            O.forced_pages(4, *bad)


@pytest.mark.parametrize("S,W", SW_CASES)
@pytest.mark.parametrize("P", [1, 3, 6, 9])
def test_selection_brute_force_with_sink_and_window(P, S, W):
    """With S first and W recent pages kept, the free pages chosen are the unique subset of the
    others in which every member beats every non-member under (score desc, index asc), and the
    output is every forced page plus that subset."""
    rng = np.random.default_rng(100 * P + 10 * S + W)
    n_forced = min(P, S + W)
    for trial in range(3):
        scores = rng.integers(-2, 3, size=P).astype(np.float64)
        for b in range(n_forced, P + 2):
            sel = O.select_pages(scores, b, S, W)
            first, last = list(range(min(S, P))), list(range(max(0, P - W), P))
            forced = sorted(set(first + last))
            others = [p for p in range(P) if p not in forced]
            k = min(b, P) - len(forced)
            winners = [sorted(forced + list(T)) for T in itertools.combinations(others, k)
                       if all((scores[x], -x) > (scores[y], -y) for x in T for y in others if y not in T)]
            assert len(winners) == 1 and winners[0] == sel and len(sel) == min(b, P)
        if P > n_forced:
            with pytest.raises(ValueError):
                O.select_pages(scores, n_forced - 1, S, W)


def test_retained_count_golden_and_closed_forms(golden_dir):
    """The printed boundary case of the retained-count rule (a ceiling, not rounding to
    nearest), then the rule's ends: r = 1 keeps all, a tiny r keeps one, the count never
    falls as r grows, and exact fractions give exact counts."""
    with open(os.path.join(golden_dir, "retained_count.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        assert O.retained_count(c["N"], c["r"]) == c["k"]
    for N in (1, 2, 13, 100, 4096):
        assert O.retained_count(N, 1.0) == N
        assert O.retained_count(N, 1e-9) == 1
        ks = [O.retained_count(N, r) for r in np.linspace(0.01, 1.0, 50)]
        assert ks == sorted(ks)
    assert O.retained_count(100, 0.05) == 5 and O.retained_count(101, 0.05) == 6
    assert O.retained_count(2048, 0.25) == 512


def test_budget_modes():
    """A fraction goes through the retained-count rule, a page count is capped at P, and both
    are raised to the always-kept set they include."""
    assert O.budget_for(13, fraction=0.1) == 2
    assert O.budget_for(13, fraction=0.1, sink_pages=2, window_pages=3) == 5
    assert O.budget_for(2200, fraction=0.05) == 110
    assert O.budget_for(50, pages=128) == 50 and O.budget_for(500, pages=128) == 128
    assert O.budget_for(500, pages=4, sink_pages=1, window_pages=10) == 11
    assert O.budget_for(3, pages=1) == 2 and O.budget_for(1, pages=1) == 1
    for bad in (dict(), dict(fraction=0.1, pages=3), dict(fraction=0.0), dict(fraction=1.5), dict(pages=0)):
        with pytest.raises(ValueError):
            O.budget_for(10, **bad)


# ------------------------------------------------------------------ latent values
def test_latent_values_are_the_key_prefix_and_match_the_inputs():
    """The latent cache's value is the first D_v dims of the key: the oracle's reading, the
    synthetic latent workload's values, and one attention check where a value column taken from
    beyond D_v would change the output."""
    w = W.reduced(5)
    keys = w.keys(0)
    v = O.latent_values(keys, w.D_v)
    assert v.shape == (keys.shape[0], 1, w.D_v) and np.array_equal(v, keys[:, :, :w.D_v])
    assert np.array_equal(v, w.values(0))
    q = w.queries()[0]
    n = int(w.seq_lens[0])
    P = -(-n // w.page_size)
    a = O.attend_pages(q, keys, v, n, w.page_size, [list(range(P))], w.dtype, 0.05)
    shifted = keys[:, :, keys.shape[2] - w.D_v:]
    b = O.attend_pages(q, keys, shifted, n, w.page_size, [list(range(P))], w.dtype, 0.05)
    assert not np.allclose(a, b)
    with pytest.raises(ValueError):
        O.latent_values(keys, keys.shape[2] + 1)


# ------------------------------------------------------------------ per-query-head selection
@pytest.mark.parametrize("seed", [0, 1])
def test_per_query_head_bound_tight_on_single_token_pages_and_dominating(seed):
    """Per query head, the bound is at or above every logit of its KV head's tokens in the page,
    equals the logit exactly on a page that holds one valid token, and its group max is the
    grouped bound."""
    rng = np.random.default_rng(300 + seed)
    H_q, H_kv, D, ps = 8, 2, 16, 16
    n = 16 * 4 + 1                                    # the tail page holds one token
    keys = _rand_keys(rng, n, H_kv, D, "bf16")
    q = W.f32_to_bf16_bits(rng.standard_normal((H_q, D)).astype(np.float32))
    kmin, kmax = O.page_summaries(keys, n, ps, "bf16")
    s = O.quest_scores_per_query_head(q, kmin, kmax, "bf16", 1.0)
    kv, qv = O.to_f64(keys, "bf16"), O.to_f64(q, "bf16")
    G = H_q // H_kv
    P = s.shape[1]
    for g in range(H_q):
        h = g // G
        for p in range(P):
            page = kv[p * ps:min((p + 1) * ps, n), h]
            logits = page @ qv[g]
            tol = 1e-12 * float(np.abs(qv[g]).sum() * np.abs(page).max())
            assert np.all(logits <= s[g, p] + tol)
        assert abs(s[g, P - 1] - float(kv[n - 1, h] @ qv[g])) <= 1e-12 * float(np.abs(qv[g]).sum() + 1)
    grouped = O.quest_scores(q, kmin, kmax, "bf16", 1.0)
    assert np.array_equal(s.reshape(H_kv, G, P).max(axis=1), grouped)


def test_per_query_head_attention_reduces_to_grouped_and_dense():
    """Each query head given its KV head's list is the grouped decode; every page for every head
    is dense attention; one head's own list is torch's attention on those tokens."""
    rng = np.random.default_rng(91)
    H_q, H_kv, D, ps, n = 8, 2, 16, 16, 16 * 7 + 5
    keys = _rand_keys(rng, n + ps, H_kv, D, "f32")
    vals = _rand_keys(rng, n + ps, H_kv, D, "f32")
    q = _rand_keys(rng, H_q, 1, D, "f32")[:, 0]
    scale = 0.25
    G = H_q // H_kv
    per_kv = [[0, 3, 7], [0, 2, 5, 7]]
    a = O.attend_pages_per_query_head(q, keys, vals, n, ps, [per_kv[g // G] for g in range(H_q)], "f32", scale)
    assert np.array_equal(a, O.attend_pages(q, keys, vals, n, ps, per_kv, "f32", scale))
    P = -(-n // ps)
    d = O.attend_pages_per_query_head(q, keys, vals, n, ps, [list(range(P))] * H_q, "f32", scale)
    assert np.array_equal(d, O.dense_attention(q, keys, vals, n, ps, "f32", scale))
    own = [[0, 1 + (g % 5), P - 1] for g in range(H_q)]
    out = O.attend_pages_per_query_head(q, keys, vals, n, ps, own, "f32", scale)
    for g in (0, 5):
        t = O.page_tokens(own[g], n, ps)
        ref = _sdpa_reference(O.to_f64(q[g:g + 1], "f32"), O.to_f64(keys[t, g // G][:, None], "f32"),
                              O.to_f64(vals[t, g // G][:, None], "f32"), scale)
        assert np.allclose(out[g], ref[0], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ S4 attention
def _sdpa_reference(q, k, v, scale):
    """torch's float64 scaled_dot_product_attention with GQA heads expanded; q [H_q, D],
    k [T, H_kv, D], v [T, H_kv, D_v]."""
    H_q, H_kv = q.shape[0], k.shape[1]
    G = H_q // H_kv
    qt = torch.from_numpy(q)[None, :, None, :]
    kt = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)[None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ps,seq_len", [(16, 16 * 6 + 5), (1, 9), (64, 64)])
def test_dense_equals_library_attention_and_full_budget_equals_dense(dtype, ps, seq_len):
    rng = np.random.default_rng(ps + seq_len)
    H_q, H_kv, D, Dv = 8, 2, 32, 24
    T = seq_len + ps
    keys = _rand_keys(rng, T, H_kv, D, dtype)
    vals = _rand_keys(rng, T, H_kv, Dv, dtype)
    q = _rand_keys(rng, H_q, 1, D, dtype)[:, 0]
    scale = 1 / math.sqrt(D)
    dense = O.dense_attention(q, keys, vals, seq_len, ps, dtype, scale)
    ref = _sdpa_reference(O.to_f64(q, dtype), O.to_f64(keys[:seq_len], dtype), O.to_f64(vals[:seq_len], dtype), scale)
    assert np.allclose(dense, ref, rtol=1e-12, atol=1e-12)
    P = -(-seq_len // ps)
    (_, _), scores, sel, out = O.decode_step(q, keys, vals, seq_len, ps, P + 3, dtype, scale)
    assert all(s == list(range(P)) for s in sel)
    assert np.array_equal(out, dense)


def test_sparse_equals_library_attention_on_selected_tokens():
    rng = np.random.default_rng(77)
    H_q, H_kv, D, ps, n = 8, 2, 16, 16, 16 * 9 + 4
    keys = _rand_keys(rng, n + ps, H_kv, D, "bf16")
    vals = _rand_keys(rng, n + ps, H_kv, D, "bf16")
    q = _rand_keys(rng, H_q, 1, D, "bf16")[:, 0]
    scale = 0.3
    (_, _), scores, sel, out = O.decode_step(q, keys, vals, n, ps, 4, "bf16", scale)
    G = H_q // H_kv
    for h in range(H_kv):
        toks = O.page_tokens(sel[h], n, ps)
        assert toks.max() < n
        ref = _sdpa_reference(O.to_f64(q[h * G:(h + 1) * G], "bf16"), O.to_f64(keys[toks, h:h + 1], "bf16"),
                              O.to_f64(vals[toks, h:h + 1], "bf16"), scale)
        assert np.allclose(out[h * G:(h + 1) * G], ref, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(9)
    D = 8
    q = rng.standard_normal(D)
    # a single token returns its value
    v = rng.standard_normal((1, 5))
    assert np.allclose(O.softmax_attention(q, rng.standard_normal((1, D)), v, 0.7), v[0], rtol=0, atol=1e-15)
    # identical keys return the mean of the values
    k = np.tile(rng.standard_normal(D), (6, 1))
    v = rng.standard_normal((6, 5))
    assert np.allclose(O.softmax_attention(q, k, v, 0.7), v.mean(0), rtol=1e-14, atol=1e-14)
    # very large logits stay finite (max subtraction)
    k = np.tile(np.full(D, 1e3), (2, 1))
    assert np.all(np.isfinite(O.softmax_attention(np.full(D, 1e3), k, v[:2], 1.0)))


def test_block_table_permutation_invariance():
    rng = np.random.default_rng(4)
    ps, n, H, D = 16, 16 * 5 + 7, 2, 8
    P = -(-n // ps)
    keys = _rand_keys(rng, P * ps, H, D, "bf16")
    for perm_seed in range(3):
        perm = np.random.default_rng(perm_seed).permutation(P + 4)[:P]
        cache = np.zeros((P + 4, ps, H, D), dtype=np.uint16)
        for p in range(P):
            cache[perm[p]] = keys[p * ps:(p + 1) * ps]
        back = O.logical_from_cache(cache, perm, n, ps)
        assert np.array_equal(back, keys[:n])


# ------------------------------------------------------------------ generator sanity
def test_workload_chunked_draws_are_consistent():
    w = W.reduced(3)
    i = 2
    n = int(w.seq_lens[i])
    full = w.keys(i)
    part = w.keys(i, 100, min(n, 5000))
    assert np.array_equal(full[100:min(n, 5000)], part)
    k, v, cu = w.packed_prefill()
    assert np.array_equal(k[cu[i]:cu[i + 1]], full)
    bt = w.block_table
    live = np.concatenate([bt[j, :w.pages(w.final_lens)[j]] for j in range(w.B)])
    assert len(set(live.tolist())) == len(live) and live.max() < w.num_blocks


# ------------------------------------------------------------------ S3 coverage mode
@pytest.fixture(scope="module")
def cov(golden_dir):
    with open(os.path.join(golden_dir, "coverage_example.json")) as f:
        return json.load(f)


def _cov_keys(cov):
    return np.log(np.asarray(cov["key_weights"], dtype=np.float64)).astype(np.float32)[:, None, None]


def test_golden_page_masses_and_coverage(cov):
    keys = _cov_keys(cov)
    q1 = _f32(cov["q_one_head"])
    m = O.page_masses(q1, keys, cov["seq_len"], cov["page_size"], "f32", 1.0)
    assert np.allclose(m[0], cov["masses_one_head"], rtol=0, atol=1e-6)
    for c, sel in cov["selected_one_head"].items():
        assert O.select_coverage(m[0], float(c), 4) == sel, c
    assert O.select_coverage(m[0], 0.9, 3) == cov["selected_one_head_b_max_3_c_0.9"]
    q2 = _f32(cov["q_two_heads"])
    g = O.group_masses(O.page_masses(q2, keys, cov["seq_len"], cov["page_size"], "f32", 1.0), 1)
    assert np.allclose(g[0], cov["group_masses_two_heads"], rtol=0, atol=1e-6)
    for c, sel in cov["selected_two_heads"].items():
        assert O.select_coverage(g[0], float(c), 4) == sel, c


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_page_masses_normalise_and_match_library_softmax(seed):
    """Each query head's page masses sum to one and equal the page sums of torch's float64
    softmax over the sequence's logits; one page holds all the mass; identical keys give masses
    proportional to the pages' token counts."""
    rng = np.random.default_rng(seed)
    ps, n, H_kv, G, D = 16, 16 * 9 + 5, 2, 3, 32
    keys = rng.standard_normal((n + 7, H_kv, D)).astype(np.float32)
    q = rng.standard_normal((H_kv * G, D)).astype(np.float32)
    scale = 1 / math.sqrt(D)
    m = O.page_masses(q, keys, n, ps, "f32", scale)
    assert np.allclose(m.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    for g in range(H_kv * G):
        logits = torch.from_numpy(keys[:n, g // G].astype(np.float64)) @ torch.from_numpy(q[g].astype(np.float64))
        w = torch.softmax(logits * scale, dim=0).numpy()
        ref = np.array([w[p * ps:(p + 1) * ps].sum() for p in range(-(-n // ps))])
        assert np.allclose(m[g], ref, rtol=1e-12, atol=1e-15)
    one = O.page_masses(q, keys, 11, ps, "f32", scale)
    assert one.shape == (H_kv * G, 1) and np.allclose(one, 1.0)
    same = np.repeat(keys[:1], n, axis=0)
    m2 = O.page_masses(q, same, n, ps, "f32", scale)
    counts = np.array([min(ps, n - p * ps) for p in range(-(-n // ps))]) / n
    assert np.allclose(m2, counts[None, :], rtol=1e-12)
    gm = O.group_masses(m, H_kv)
    for h in range(H_kv):
        assert np.array_equal(gm[h], m[h * G:(h + 1) * G].max(axis=0))
    assert np.array_equal(O.group_masses(m, H_kv * G), m)


@pytest.mark.parametrize("P", [1, 2, 4, 7, 9])
def test_coverage_selection_brute_force(P):
    """Against subset enumeration: the selection holds the always-kept pages; it reaches the
    target unless the b_max cap or the pages run out; no smaller set holding the always-kept
    pages reaches the target; and its other pages beat every page left out under
    (mass desc, index asc), ties included."""
    rng = np.random.default_rng(50 + P)
    for trial in range(12):
        if trial % 3 == 2:
            mass = rng.integers(0, 4, size=P).astype(np.float64)   # ties and zero masses
        else:
            mass = rng.dirichlet(np.ones(P))
        for S, Wn in ((1, 1), (0, 1), (2, 1)):
            forced = sorted(set(range(min(S, P))) | set(range(max(0, P - Wn), P)))
            others = [p for p in range(P) if p not in forced]
            for c in (0.05, 0.5, 0.9, 0.999, 1.0):
                target = c * mass.sum()
                for b_max in range(len(forced), P + 1):
                    sel = O.select_coverage(mass, c, b_max, S, Wn)
                    assert sel == sorted(set(sel)) and set(forced) <= set(sel) and len(sel) <= b_max
                    got = mass[sel].sum()
                    assert got >= target or len(sel) == b_max or len(sel) == P
                    need = None
                    for k in range(len(others) + 1):
                        if any(mass[forced].sum() + mass[list(sub)].sum() >= target
                               for sub in itertools.combinations(others, k)):
                            need = k
                            break
                    if need is not None:
                        assert len(sel) - len(forced) == min(need, b_max - len(forced))
                    chosen = [p for p in sel if p not in forced]
                    left = [p for p in others if p not in chosen]
                    assert all((mass[x], -x) > (mass[y], -y) for x in chosen for y in left)


# ------------------------------------------------------------------ S1 / S2 mean-std summaries, Gaussian score
@pytest.fixture(scope="module")
def msx(golden_dir):
    with open(os.path.join(golden_dir, "mean_std_example.json")) as f:
        return json.load(f)


def test_golden_mean_std_and_gaussian_score(msx):
    keys = _f32(msx["keys"])[:, None, :]
    mean, std = O.page_mean_std(keys, msx["seq_len"], msx["page_size"], "f32")
    assert np.array_equal(mean[:, 0], np.asarray(msx["mean"], dtype=np.float64))
    assert np.array_equal(std[:, 0], np.asarray(msx["std"], dtype=np.float64))
    q = _f32(msx["q"])
    per_head = O.gaussian_scores(q, np.repeat(mean, 2, axis=1), np.repeat(std, 2, axis=1), "f32", 1.0, msx["z"])
    assert np.allclose(per_head, msx["score_per_query_head_unscaled"], rtol=0, atol=1e-12)
    s = O.gaussian_scores(q, mean, std, "f32", 1.0 / math.sqrt(2.0), msx["z"])
    assert np.allclose(s[0] * math.sqrt(2.0), msx["group_score_unscaled"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mean_std_closed_forms_and_parallel_merge(dtype):
    """Two tokens: mean (a + b) / 2, std |a - b| / 2; a constant shift moves the mean and keeps
    the std; a scale scales both; and the statistics of a page equal the merge of its two
    halves' by the parallel-variance formula (n, mean, n * var) of Chan, Golub and LeVeque;
    tokens past seq_len are ignored."""
    rng = np.random.default_rng(3)
    ps, n, H, D = 16, 16 * 4 + 6, 2, 8
    keys = _rand_keys(rng, n + 10, H, D, dtype)
    mean, std = O.page_mean_std(keys, n, ps, dtype)
    v = O.to_f64(keys, dtype)
    two = O.page_mean_std(keys[:2], 2, 2, dtype)
    assert np.allclose(two[0][0], (v[0] + v[1]) / 2, rtol=0, atol=1e-15)
    assert np.allclose(two[1][0], np.abs(v[0] - v[1]) / 2, rtol=1e-14, atol=1e-15)
    # bf16-valued keys held as fp32: adding 0.5 or scaling by -4 is exact on them
    f = O.to_f64(W.f32_to_bf16_bits(rng.standard_normal((n, H, D)).astype(np.float32)), "bf16").astype(np.float32)
    m2, s2 = O.page_mean_std(f + np.float32(0.5), n, ps, "f32")
    m1, s1 = O.page_mean_std(f, n, ps, "f32")
    assert np.allclose(m2, m1 + 0.5, rtol=0, atol=1e-12) and np.allclose(s2, s1, rtol=1e-9, atol=1e-12)
    m3, s3 = O.page_mean_std(f * np.float32(-4.0), n, ps, "f32")
    assert np.allclose(m3, -4 * m1, rtol=1e-12, atol=1e-12) and np.allclose(s3, 4 * s1, rtol=1e-12, atol=1e-12)
    for p in range(mean.shape[0]):
        page = v[p * ps:min((p + 1) * ps, n)]
        a, b = page[:len(page) // 2], page[len(page) // 2:]
        if len(a) == 0:
            continue
        na, nb = len(a), len(b)
        ma, mb = a.mean(axis=0), b.mean(axis=0)
        Ma, Mb = ((a - ma) ** 2).sum(axis=0), ((b - mb) ** 2).sum(axis=0)
        delta = mb - ma
        M = Ma + Mb + delta ** 2 * na * nb / (na + nb)
        assert np.allclose(mean[p], ma + delta * nb / (na + nb), rtol=1e-12, atol=1e-14)
        assert np.allclose(std[p], np.sqrt(M / (na + nb)), rtol=1e-9, atol=1e-12)
    junk = keys.copy()
    junk[n:] = _rand_keys(rng, 10, H, D, dtype)
    mj, sj = O.page_mean_std(junk, n, ps, dtype)
    assert np.array_equal(mj, mean) and np.array_equal(sj, std)


@pytest.mark.parametrize("seed", [0, 1])
def test_gaussian_score_reductions(seed):
    """z = 0 gives scale times the page's average logit (brute force over its tokens); a page
    whose keys vary in one dimension only has logit std |q_d| std_d exactly, so z = 1 gives the
    mean plus the logits' own population std; single-token pages give the exact logit and the
    selection equals the textbook top-k of the logits."""
    rng = np.random.default_rng(seed)
    ps, P, H_kv, G, D = 8, 12, 2, 2, 16
    keys = rng.standard_normal((P * ps, H_kv, D)).astype(np.float32)
    q = rng.standard_normal((H_kv * G, D)).astype(np.float32)
    scale = 1 / math.sqrt(D)
    mean, std = O.page_mean_std(keys, P * ps, ps, "f32")
    s0 = O.gaussian_scores(q, mean, std, "f32", scale, 0.0)
    for h in range(H_kv):
        for p in range(P):
            toks = keys[p * ps:(p + 1) * ps, h].astype(np.float64)
            avg = max((toks @ q[g].astype(np.float64)).mean() for g in range(h * G, (h + 1) * G))
            assert abs(s0[h, p] - scale * avg) <= 1e-12 * (1 + abs(avg))
    one = np.repeat(keys[:1], P * ps, axis=0).copy()
    one[:, :, 3] = rng.standard_normal((P * ps, H_kv)).astype(np.float32)
    mean1, std1 = O.page_mean_std(one, P * ps, ps, "f32")
    s1 = O.gaussian_scores(q, mean1, std1, "f32", 1.0, 1.0)
    for h in range(H_kv):
        for p in range(P):
            toks = one[p * ps:(p + 1) * ps, h].astype(np.float64)
            best = max((toks @ q[g].astype(np.float64)).mean() + (toks @ q[g].astype(np.float64)).std()
                       for g in range(h * G, (h + 1) * G))
            assert abs(s1[h, p] - best) <= 1e-9 * (1 + abs(best))
    single = rng.standard_normal((P, 1, D)).astype(np.float32)
    q1 = rng.standard_normal((1, D)).astype(np.float32)
    m, sd = O.page_mean_std(single, P, 1, "f32")
    assert np.all(sd == 0)
    sc = O.gaussian_scores(q1, m, sd, "f32", 1.0, 3.0)[0]
    logits = single[:, 0].astype(np.float64) @ q1[0].astype(np.float64)
    assert np.allclose(sc, logits, rtol=1e-12, atol=1e-12)
    b = 6
    sel = O.select_pages(sc, b)
    top = torch.topk(torch.from_numpy(logits[1:P - 1]), b - 2).indices.numpy() + 1
    assert sel == sorted([0, P - 1] + [int(x) for x in top])
