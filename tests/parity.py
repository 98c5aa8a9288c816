"""Comparison rules shared by the GPU parity tests (CUDA path vs the fp64 oracle).

  * summaries, cache contents and selected page ids: bit-exact, except that selected ids
    may differ at the cutoff when every differing page's oracle score is within 1e-6
    relative of the oracle's cutoff score (a near tie fp32 accumulation may resolve
    differently); such units are reported and the output check then feeds the GPU's ids
    to the oracle's attention.
  * bf16 outputs: max-abs <= 2e-2 and mean-abs <= 2e-3 against the fp64 oracle.
  * fp32 outputs: per output row, max-abs error / max-abs oracle value <= 1e-5.
  * page scores (fp32 vs fp64): |gpu - oracle| <= 2e-6 * sum_d |q_d| * max(|kmin_d|, |kmax_d|)
    (max over the group), the bound on fp32 rounding of a D-term sum with one rounding
    per term at 2^-24 relative, with a margin.
"""
from __future__ import annotations

import os

import numpy as np

import oracle as O

NEAR_TIE_REL = 1e-6

# Every selection comparison of the session: units compared, and the near ties accepted at the
# cutoff with where they occurred (the test id and the differing pages with their oracle scores
# relative to the cutoff). tests/conftest.py prints the tally in the terminal summary.
SELECTION_LOG = {"units": 0, "near_ties": []}


def _log(near: bool, diff=(), scores=None, cut=None):
    SELECTION_LOG["units"] += 1
    if near:
        where = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        rel = [float(abs(scores[p] - cut) / abs(cut)) if cut else 0.0 for p in sorted(diff)]
        SELECTION_LOG["near_ties"].append({"test": where, "pages": sorted(int(p) for p in diff), "rel_to_cutoff": rel})
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
F32_ROW_REL = 1e-5


def compare_selection(gpu_row: np.ndarray, scores: np.ndarray, budget: int, sink_pages: int = 1,
                      window_pages: int = 1, near_rel: float = NEAR_TIE_REL):
    """gpu_row: int32 [b_max] (ascending ids, -1 padded); scores: oracle fp64 [P]. near_rel: the
    near-tie band relative to the cutoff score (1e-6 for the bound; wider for scores built from
    fp32 statistics). Returns (ok, near_tie, gpu_ids, oracle_ids)."""
    ref = O.select_pages(scores, budget, sink_pages, window_pages)
    got = [int(x) for x in gpu_row if x >= 0]
    pad_ok = all(x < 0 for x in gpu_row[len(got):])
    if got == ref and pad_ok:
        _log(False)
        return True, False, got, ref
    if len(got) != len(ref) or not pad_ok or got != sorted(set(got)):
        return False, False, got, ref
    cut = O.cutoff_score(scores, budget, sink_pages, window_pages)
    diff = set(got) ^ set(ref)
    if cut is None:
        return False, False, got, ref
    near = all(abs(scores[p] - cut) <= near_rel * abs(cut) for p in diff)
    forced_ok = set(O.forced_pages(len(scores), sink_pages, window_pages)) <= set(got)
    if near and forced_ok:
        _log(True, diff, scores, cut)
    return (near and forced_ok), near, got, ref


MASS_REL = 1e-5  # page masses (fp32 vs fp64), relative to the unit's largest mass; sums: to its total


def compare_coverage(gpu_row: np.ndarray, mass: np.ndarray, coverage: float, b_max: int, sink_pages: int = 1,
                     window_pages: int = 1):
    """Adaptive coverage: gpu_row must be a valid nucleus under the oracle's fp64 masses [P], up
    to fp32 rounding of the masses (MASS_REL): ascending, -1 padded, the always-kept pages
    included, at most b_max pages; every other page chosen outweighs every page left out (up to
    the tolerance); the coverage target is reached unless b_max or the pages run out; and dropping
    the lightest chosen page would fall short of it. Returns (ok, same_as_oracle, gpu, oracle)."""
    ref = O.select_coverage(mass, coverage, b_max, sink_pages, window_pages)
    got = [int(x) for x in gpu_row if x >= 0]
    pad_ok = all(x < 0 for x in gpu_row[len(got):])
    P = len(mass)
    if got == ref and pad_ok:
        return True, True, got, ref
    forced = O.forced_pages(P, sink_pages, window_pages)
    if not pad_ok or got != sorted(set(got)) or not set(forced) <= set(got) or len(got) > b_max:
        return False, False, got, ref
    if any(p < 0 or p >= P for p in got):
        return False, False, got, ref
    tol = MASS_REL * float(mass.max())
    tol_sum = MASS_REL * float(mass.sum())
    chosen = [p for p in got if p not in forced]
    left = [p for p in range(P) if p not in got]
    if chosen and left and max(mass[left]) > min(mass[chosen]) + tol:
        return False, False, got, ref
    target = coverage * float(mass.sum())
    have = float(mass[got].sum())
    if have < target - tol_sum and len(got) < b_max and left:
        return False, False, got, ref
    if chosen and have - float(min(mass[chosen])) >= target + tol_sum:
        return False, False, got, ref
    return True, False, got, ref


def score_tolerance(q: np.ndarray, kmin: np.ndarray, kmax: np.ndarray, dtype: str, scale: float) -> np.ndarray:
    """Per (kv head, page) bound on fp32 accumulation error of the page score."""
    qv, lo, hi = O.to_f64(q, dtype), O.to_f64(kmin, dtype), O.to_f64(kmax, dtype)
    H_q = qv.shape[0]
    P, H_kv, D = lo.shape
    G = H_q // H_kv
    mag = np.maximum(np.abs(lo), np.abs(hi))
    out = np.empty((H_kv, P))
    for h in range(H_kv):
        out[h] = np.max(np.abs(qv[h * G:(h + 1) * G]) @ mag[:, h, :].T, axis=0)
    return 2e-6 * out * scale + 1e-30


def check_output(gpu: np.ndarray, ref: np.ndarray, dtype: str):
    """Raises AssertionError with the measured errors when out of tolerance."""
    err = np.abs(gpu.astype(np.float64) - ref)
    if dtype == "bf16":
        mx, mean = float(err.max()), float(err.mean())
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, f"max-abs {mx:.3e} mean-abs {mean:.3e}"
        return mx, mean
    rows = err.reshape(-1, err.shape[-1]).max(axis=1) / np.maximum(np.abs(ref).reshape(-1, ref.shape[-1]).max(axis=1),
                                                                     1e-300)
    assert rows.max() <= F32_ROW_REL, f"row-relative {rows.max():.3e}"
    return float(rows.max()), float(err.mean())
