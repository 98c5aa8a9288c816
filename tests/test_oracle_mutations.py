"""The oracle's pins catch plausible mistakes (CPU only).

Each test swaps one oracle function for a copy with a typical slip (a dropped term, a wrong
reduction, a tie broken the other way, the tail not forced, tokens past seq_len counted, signed
zeros confused, the scale left out) and checks that a pin of test_oracle_pins.py then fails. The
mistakes are planted in the oracle only, on the CPU; nothing here touches a GPU.
"""
import numpy as np
import pytest

import oracle as O
import oracle.psk_oracle as OP
import test_oracle_pins as PINS

ORIG = {name: getattr(OP, name) for name in ("quest_scores", "select_pages", "page_summaries", "softmax_attention",
                                             "forced_pages", "retained_count", "quest_scores_per_query_head",
                                             "cutoff_score", "page_masses", "select_coverage", "page_mean_std",
                                             "gaussian_scores")}


@pytest.fixture
def plant(monkeypatch):
    def _plant(name, fn):
        monkeypatch.setattr(OP, name, fn)  # calls inside the oracle module
        monkeypatch.setattr(O, name, fn)   # calls through the package, as the pins make them
    return _plant


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


# ---- planted mistakes ---------------------------------------------------------------------
def _quest_kmax_only(q, kmin, kmax, dtype, scale):  # drops the q * kmin term
    return ORIG["quest_scores"](q, kmax, kmax, dtype, scale)


def _quest_group_mean(q, kmin, kmax, dtype, scale):  # mean over the GQA group instead of max
    qv, lo, hi = O.to_f64(q, dtype), O.to_f64(kmin, dtype), O.to_f64(kmax, dtype)
    G = qv.shape[0] // lo.shape[1]
    per = [[np.maximum(qv[h * G + j] * lo[:, h, :], qv[h * G + j] * hi[:, h, :]).sum(axis=1) for j in range(G)]
           for h in range(lo.shape[1])]
    return np.stack([np.mean(p, axis=0) for p in per]) * scale


def _quest_no_scale(q, kmin, kmax, dtype, scale):  # forgets 1/sqrt(D)
    return ORIG["quest_scores"](q, kmin, kmax, dtype, 1.0)


def _select_ties_high(scores, budget, sink_pages=1, window_pages=1):  # ties go to the higher page index
    P = len(scores)
    forced = O.forced_pages(P, sink_pages, window_pages)
    count = min(budget, P)
    ranked = sorted((p for p in range(P) if p not in forced), key=lambda p: (-float(scores[p]), -p))
    return sorted(forced + ranked[:count - len(forced)])


def _select_tail_not_forced(scores, budget, sink_pages=1, window_pages=1):  # only the sink is forced
    P = len(scores)
    count = min(budget, P)
    ranked = sorted(range(1, P), key=lambda p: (-float(scores[p]), p))
    return sorted([0] + ranked[:count - 1])


def _forced_window_of_one(P, sink_pages=1, window_pages=1):  # window_pages read as 1
    return ORIG["forced_pages"](P, sink_pages, 1)


def _retained_round_nearest(N, r):  # rounds N * r to nearest instead of the ceiling
    return min(N, max(1, int(round(N * r))))


def _per_query_head_wrong_kv_head(q, kmin, kmax, dtype, scale):  # query head g read KV head g % H_kv
    H_q, H_kv = q.shape[0], kmin.shape[1]
    order = [(g % H_kv) * (H_q // H_kv) + g // H_kv for g in range(H_q)]
    return ORIG["quest_scores_per_query_head"](q[order], kmin, kmax, dtype, scale)[np.argsort(order)]


def _summaries_whole_pages(keys, seq_len, page_size, dtype):  # counts the tail page's junk rows
    P = -(-seq_len // page_size)
    return ORIG["page_summaries"](keys, min(len(keys), P * page_size), page_size, dtype)


def _summaries_plain_minmax(keys, seq_len, page_size, dtype):  # -0.0 and +0.0 compare equal
    v = O.to_f64(keys, dtype)[:seq_len]
    P = -(-seq_len // page_size)
    lo = np.stack([v[p * page_size:(p + 1) * page_size].min(axis=0) for p in range(P)])
    hi = np.stack([v[p * page_size:(p + 1) * page_size].max(axis=0) for p in range(P)])
    return O.exact_to_storage(lo, dtype), O.exact_to_storage(hi, dtype)


def _attention_unscaled(q, k, v, scale):  # logits without the scale
    return ORIG["softmax_attention"](q, k, v, 1.0)


def _cutoff_one_too_far(scores, budget, sink_pages=1, window_pages=1):  # the k_free-th ranked page, one past the cut
    P = len(scores)
    forced = O.forced_pages(P, sink_pages, window_pages)
    k_free = min(budget, P) - len(forced)
    if min(budget, P) >= P or k_free <= 0:
        return None
    ranked = sorted((p for p in range(P) if p not in forced), key=lambda p: (-float(scores[p]), p))
    return float(scores[ranked[min(k_free, len(ranked) - 1)]])


def _masses_per_page_softmax(q, keys, seq_len, page_size, dtype, scale):  # normalised within each page
    m = ORIG["page_masses"](q, keys, seq_len, page_size, dtype, scale)
    P = m.shape[1]
    out = np.empty_like(m)
    qv, k = O.to_f64(q, dtype), O.to_f64(keys[:seq_len], dtype)
    G = qv.shape[0] // keys.shape[1]
    for g in range(qv.shape[0]):
        for p in range(P):
            lg = scale * (k[p * page_size:min((p + 1) * page_size, seq_len), g // G] @ qv[g])
            out[g, p] = 1.0 if len(lg) else 0.0
    return out


def _coverage_ignores_forced_mass(mass, coverage, b_max, sink_pages=1, window_pages=1):  # forced mass not counted
    P = len(mass)
    forced = O.forced_pages(P, sink_pages, window_pages)
    target, have = coverage * float(mass.sum()), 0.0
    chosen = []
    for p in sorted((p for p in range(P) if p not in forced), key=lambda p: (-float(mass[p]), p)):
        if have >= target or len(forced) + len(chosen) >= b_max:
            break
        chosen.append(p)
        have += float(mass[p])
    return sorted(forced + chosen)


def _std_sample_divisor(keys, seq_len, page_size, dtype):  # n - 1 instead of n
    mean, std = ORIG["page_mean_std"](keys, seq_len, page_size, dtype)
    P = mean.shape[0]
    n = np.array([min(page_size, seq_len - p * page_size) for p in range(P)], dtype=np.float64)
    fix = np.sqrt(n / np.maximum(n - 1, 1))[:, None, None]
    return mean, std * fix


def _gaussian_without_spread(q, mean, std, dtype, scale, z):  # the z * std term dropped
    return ORIG["gaussian_scores"](q, mean, std, dtype, scale, 0.0)


# ---- each one is caught -------------------------------------------------------------------
def test_dropped_kmin_term_is_caught(plant):
    plant("quest_scores", _quest_kmax_only)
    _fails(PINS.test_bound_dominates_every_token_logit, 0)


def test_group_mean_instead_of_max_is_caught(plant):
    plant("quest_scores", _quest_group_mean)
    _fails(PINS.test_bound_group_max_and_scale)


def test_missing_scale_is_caught(plant):
    plant("quest_scores", _quest_no_scale)
    _fails(PINS.test_bound_group_max_and_scale)


def test_ties_to_higher_index_are_caught(plant):
    plant("select_pages", _select_ties_high)
    _fails(PINS.test_selection_tie_lower_index_wins_on_copied_page)


def test_tail_not_forced_is_caught(plant):
    plant("select_pages", _select_tail_not_forced)
    _fails(PINS.test_selection_brute_force_subsets, 5)


def test_tokens_past_seq_len_in_summaries_are_caught(plant):
    plant("page_summaries", _summaries_whole_pages)
    _fails(PINS.test_summary_bounds_attained_and_tail_masked, "f32", 16, 16 * 5 + 3)


def test_signed_zero_order_is_caught(plant):
    plant("page_summaries", _summaries_plain_minmax)
    _fails(PINS.test_summary_signed_zero_order)


def test_unscaled_attention_is_caught(plant):
    plant("softmax_attention", _attention_unscaled)
    _fails(PINS.test_dense_equals_library_attention_and_full_budget_equals_dense, "f32", 16, 16 * 6 + 5)


def test_window_of_one_is_caught(plant):
    plant("forced_pages", _forced_window_of_one)
    _fails(PINS.test_selection_brute_force_with_sink_and_window, 6, 1, 3)


def test_fraction_rounded_to_nearest_is_caught(plant, golden_dir):
    plant("retained_count", _retained_round_nearest)
    _fails(PINS.test_retained_count_golden_and_closed_forms, golden_dir)


def test_per_query_head_wrong_kv_head_is_caught(plant):
    plant("quest_scores_per_query_head", _per_query_head_wrong_kv_head)
    _fails(PINS.test_per_query_head_bound_tight_on_single_token_pages_and_dominating, 0)


def test_cutoff_one_place_too_far_is_caught(plant, golden_dir):
    plant("cutoff_score", _cutoff_one_too_far)
    import json
    import os
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        ex = json.load(f)
    _fails(PINS.test_golden_cutoff_score, ex)
    _fails(PINS.test_cutoff_score_is_the_weakest_winner_by_enumeration, 8)


def test_masses_normalised_per_page_are_caught(plant):
    plant("page_masses", _masses_per_page_softmax)
    _fails(PINS.test_page_masses_normalise_and_match_library_softmax, 0)


def test_coverage_ignoring_forced_mass_is_caught(plant, golden_dir):
    plant("select_coverage", _coverage_ignores_forced_mass)
    import json
    import os
    with open(os.path.join(golden_dir, "coverage_example.json")) as f:
        cov = json.load(f)
    _fails(PINS.test_golden_page_masses_and_coverage, cov)
    _fails(PINS.test_coverage_selection_brute_force, 7)


def test_sample_std_divisor_is_caught(plant):
    plant("page_mean_std", _std_sample_divisor)
    _fails(PINS.test_mean_std_closed_forms_and_parallel_merge, "f32")


def test_gaussian_spread_dropped_is_caught(plant, golden_dir):
    plant("gaussian_scores", _gaussian_without_spread)
    import json
    import os
    with open(os.path.join(golden_dir, "mean_std_example.json")) as f:
        msx = json.load(f)
    _fails(PINS.test_golden_mean_std_and_gaussian_score, msx)
    _fails(PINS.test_gaussian_score_reductions, 0)
