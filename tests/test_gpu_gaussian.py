"""GPU parity of the mean / std page summaries and the Gaussian page score against the oracle.

The fp32 mean / std store kept by psk_kv_append_and_summarize_ex is checked against
oracle.page_mean_std after the prefill and after every decode append (the refresh recomputes
touched pages from their tokens, so it equals a rebuild); the Gaussian scores against
oracle.gaussian_scores on the oracle's own statistics (within an fp32 bound); the selected ids
with a near-tie band for fp32 statistics; and the sparse decode over those pages against the
oracle's attention.

Tolerances: a page statistic differs from fp64 by fp32 rounding of at most 64 terms, within
1e-5 of the page's largest |key| (plus 1e-30); a score by at most 1e-5 of
scale * sum_d |q_d| (|mean_d| + z std_d), max over the group; selected ids may differ from the
oracle's only where the oracle's scores lie within 1e-5 relative of its cutoff (reported).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from parity import check_output, compare_selection

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import page_sparse_kv_gb300 as psk  # noqa: E402
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload  # noqa: E402

STAT_REL, SCORE_REL, NEAR_REL = 1e-5, 1e-5, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from page_sparse_kv_gb300.build import build
    build()


def _custom(seq_lens, budgets, ps=16, dtype="bf16", H_q=8, H_kv=2, D=128, seed=31, appends=0):
    return W.Workload("gauss", seed, dtype, B=len(seq_lens), H_q=H_q, H_kv=H_kv, D=D, D_v=D, page_size=ps,
                      seq_lens=seq_lens, budgets=budgets, n_hot=4, hot_rule="random", pool_slack=3, appends=appends)


def _stats_from_prefill(w, cache):
    """Re-appends every sequence's prompt in place with the mean / std store only."""
    stats = torch.zeros(w.num_blocks, w.H_kv, 2, w.D, dtype=torch.float32, device="cuda")
    k, v, _ = w.packed_prefill(list(range(w.B)))
    cu = np.zeros(w.B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(w.seq_lens.astype(np.int64))
    psk.kv_append_and_summarize_ex(cache.layout, to_torch(k, w.dtype).cuda(), to_torch(v, w.dtype).cuda(),
                                   torch.zeros(w.B, dtype=torch.int32, device="cuda"), torch.from_numpy(cu).cuda(),
                                   int(w.seq_lens.max()), cache.k_cache, cache.v_cache, None, stats,
                                   cache.block_table, cache.ws)
    return stats


def _check_stats(w, stats_np, i, keys, n):
    mean, std = O.page_mean_std(keys, n, w.page_size, w.dtype)
    P = mean.shape[0]
    blocks = w.block_table[i, :P]
    v = O.to_f64(keys[:n], w.dtype)
    for p in range(P):
        page = v[p * w.page_size:min((p + 1) * w.page_size, n)]
        tol = STAT_REL * np.abs(page).max(axis=0) + 1e-30
        assert np.all(np.abs(stats_np[blocks[p], :, 0] - mean[p]) <= tol), f"seq {i} page {p}: mean"
        assert np.all(np.abs(stats_np[blocks[p], :, 1] - std[p]) <= tol), f"seq {i} page {p}: std"
    return mean, std


def _score_select_and_check(w, cache, stats, q_np, z, keys_of, lens):
    L = cache.layout
    q = to_torch(q_np, w.dtype).cuda()
    scores = torch.full((w.B, w.H_kv, w.max_pages), float("nan"), device="cuda")
    sel = torch.full((w.B, w.H_kv, cache.b_max), -7, dtype=torch.int32, device="cuda")
    psk.page_score_select_gaussian(L, q, stats, cache.block_table, cache.seq_lens, cache.b_max, cache.scale, z, sel,
                                   cache.ws, budgets=dev_budgets(w), scores_out=scores)
    out = cache.sparse_decode(q, sel)
    torch.cuda.synchronize()
    assert psk.get_device_status(cache.ws) == 0
    stats_np, sc_np, sel_np = stats.cpu().numpy(), scores.cpu().numpy(), sel.cpu().numpy()
    out_np = from_torch(out.float(), "f32")
    scale = 1.0 / math.sqrt(w.D)
    G = w.H_q // w.H_kv
    for i in range(w.B):
        n = lens[i]
        keys, vals = keys_of(i)
        mean, std = _check_stats(w, stats_np, i, keys, n)
        P = mean.shape[0]
        s_ref = O.gaussian_scores(q_np[i], mean, std, w.dtype, scale, z)
        qv = np.abs(O.to_f64(q_np[i], w.dtype))
        for h in range(w.H_kv):
            mag = np.max(qv[h * G:(h + 1) * G] @ (np.abs(mean[:, h, :]) + z * std[:, h, :]).T, axis=0)
            assert np.all(np.abs(sc_np[i, h, :P] - s_ref[h]) <= SCORE_REL * mag * scale + 1e-30), f"seq {i} head {h}"
        use = []
        for h in range(w.H_kv):
            ok, _, got, ref = compare_selection(sel_np[i, h], s_ref[h], int(w.budgets[i]), near_rel=NEAR_REL)
            assert ok, f"seq {i} head {h}: selected {got} vs oracle {ref}"
            use.append(got)
        check_output(out_np[i], O.attend_pages(q_np[i], keys, vals, n, w.page_size, use, w.dtype, scale), w.dtype)


@pytest.mark.parametrize("case", [
    dict(seq_lens=[16 * 300 + 5, 16 * 77, 16 * 40 + 9, 33, 1], budgets=[40, 9, 12, 3, 2], z=1.5),
    dict(seq_lens=[16 * 90 + 3, 300], budgets=[10, 5], z=2.0, dtype="f32", D=64, H_q=4, H_kv=1),
    dict(seq_lens=[16 * 70 + 3, 500], budgets=[9, 4], z=0.0, D=64, H_q=8, H_kv=4),
    dict(seq_lens=[64 * 40 + 33, 64 * 9], budgets=[7, 3], z=2.5, ps=64, H_q=16, H_kv=8),
])
def test_gaussian_summaries_and_selection(case):
    extra = {k: case[k] for k in ("ps", "dtype", "D", "H_q", "H_kv") if k in case}
    w = _custom(case["seq_lens"], case["budgets"], **extra)
    cache = upload(w)
    stats = _stats_from_prefill(w, cache)
    lens = [int(x) for x in w.seq_lens]
    _score_select_and_check(w, cache, stats, w.queries(), case["z"], lambda i: (w.keys(i), w.values(i)), lens)


def test_gaussian_summaries_follow_decode_appends():
    """Decode appends with both stores: the touched page's mean / std equal the oracle's rebuild
    after every token (pages fill up and new pages start), and the step stays oracle-matched."""
    w = _custom([16 * 30 + 13, 16 * 12], [8, 5], appends=6)  # block-table rows hold the appended pages
    cache = upload(w)
    stats = _stats_from_prefill(w, cache)
    rng = np.random.default_rng(4)
    K = [w.keys(i) for i in range(w.B)]
    V = [w.values(i) for i in range(w.B)]
    lens = [int(x) for x in w.seq_lens]
    for step in range(6):
        k_new = W.f32_to_bf16_bits(rng.standard_normal((w.B, w.H_kv, w.D)).astype(np.float32))
        v_new = W.f32_to_bf16_bits(rng.standard_normal((w.B, w.H_kv, w.D)).astype(np.float32))
        start = torch.tensor(lens, dtype=torch.int32, device="cuda")
        cu = torch.arange(w.B + 1, dtype=torch.int32, device="cuda")
        psk.kv_append_and_summarize_ex(cache.layout, to_torch(k_new, w.dtype).cuda(), to_torch(v_new, w.dtype).cuda(),
                                       start, cu, 1, cache.k_cache, cache.v_cache, cache.summaries, stats,
                                       cache.block_table, cache.ws)
        for i in range(w.B):
            K[i] = np.concatenate([K[i], k_new[i][None]])
            V[i] = np.concatenate([V[i], v_new[i][None]])
            lens[i] += 1
        cache.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        stats_np = stats.cpu().numpy()
        for i in range(w.B):
            _check_stats(w, stats_np, i, K[i], lens[i])
    _score_select_and_check(w, cache, stats, w.queries(3), 1.5, lambda i: (K[i], V[i]), lens)
