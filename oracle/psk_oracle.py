"""Plain fp64 CPU oracle for page-selective sparse paged decode attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` may import this module. The product
path (the CUDA library and its Python binding) never calls it and shares no
code with it.

Every step is the literal definition, evaluated in float64 from the exact
stored input values (bf16 bit patterns or fp32), with no blocking, split-K,
online softmax or algebraic rewriting:

  S1 page summaries   -- elementwise k_min / k_max of each page's keys per KV head
                         (EntmaxKV README, introduction: pages are scored from
                         per-page key statistics, "min/max for top-k"; repository
                         layout, kernels/page_metadata.py "per-page k_min / k_max
                         refresh"). Tokens at or past seq_len are not part of any
                         page's summary.
  S2 page score       -- Quest-style upper bound sum_d max(q_d*kmin_d, q_d*kmax_d)
                         (EntmaxKV README, "Two selection strategies: Top-k";
                         kernels/page_criticality.py), combined over the query heads
                         of a GQA group by max (LOCKS PKG-INFO, configuration table,
                         GQA group combine option `max`), times 1/sqrt(D).
  S3 select           -- static top-b pages per (sequence, KV head) (LOCKS PKG-INFO,
                         "How it works", Selection (Stage A)); the sink page 0 and
                         the current tail page are always kept and counted inside b
                         (LOCKS "Results" preamble: "sink + recent counted inside b";
                         EntmaxKV "Top-k": the budget includes the always-attended
                         tail page); ties go to the lower logical page index. The
                         always-kept set generalises to the first sink_pages and the
                         last window_pages pages (LOCKS configuration table), and b
                         may come from a fraction of the pages or a fixed page count
                         (same table; the fraction rounds by the retained-count rule
                         of the vllm-rlt pull request #157 discussion).
  S2 Gaussian score   -- per-page key mean / std (EntmaxKV "mean/std for Gaussian") and the
                         estimated page maximum q.mean + z * sqrt(sum (q std)^2), max over the
                         group, times scale.
  S3 coverage mode    -- adaptive per-head nucleus coverage over exact page masses (LOCKS
                         configuration table `coverage`; AMASS "Key AmassConfig fields"): the
                         softmax mass of every page, max over the GQA group, and the fewest
                         highest-mass pages that, with the always-kept ones, reach a fraction of
                         the total mass.
  S4 attention        -- exact softmax attention over the selected pages' tokens
                         only (EntmaxKV introduction: "the attention is exact over
                         that selection"; LOCKS "How it works", Sparse decode), the
                         tail page masked at seq_len.

Parity pins for every function live in tests/test_oracle_pins.py. Readings of
points the pages leave open:
  * a page's "tail" is page ceil(seq_len / page_size) - 1, the page that holds
    token seq_len - 1;
  * the selected count is min(b, P); with P == 1 the sink is the tail;
  * overlapping sink and window sets count once; a budget below the forced set's size is
    an error, and a budget mode's result is raised to that size;
  * min / max order signed zeros as -0.0 < +0.0 (IEEE 754 totalOrder on non-NaN);
  * ties in the page score (including -0.0 vs +0.0) go to the lower page index;
  * the scale 1/sqrt(D) is applied after the group max and is the same scale
    used for the attention logits;
  * for a latent (MLA) cache the value is the first D_v dims of the latent key;
  * mean / std summaries: population standard deviation (divisor n) over the page's valid
    tokens; the Gaussian score treats the key dimensions as independent and its estimated
    maximum is mean + z * std with z chosen by the caller, ranked top-b like the bound (the
    entmax threshold the EntmaxKV selector solves for is out of scope);
  * coverage: a page's mass is its exact softmax mass for a query head over every token of the
    sequence; a KV head's page mass is the max over its group's query heads; the always-kept
    pages are selected and their mass counts toward the target, which is the coverage fraction
    of the unit's total page mass; the other pages join in (mass desc, index asc) order until
    the target is reached, and the selection holds at most b_max pages.
"""
from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------------
# storage <-> float64
# ----------------------------------------------------------------------------------
def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements (fp32 values, or bf16 bit patterns as uint16)."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def exact_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Store float64 values that are exactly representable in ``dtype`` (e.g. a min or max
    of stored values). Raises if a value would round."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), x, equal_nan=False):
        raise ValueError("value not representable in fp32")
    if dtype == "f32":
        return f
    bits = f.view(np.uint32)
    if np.any(bits & np.uint32(0xFFFF)):
        raise ValueError("value not representable in bf16")
    return (bits >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------------
# S1: page summaries
# ----------------------------------------------------------------------------------
def _signed_zero_fix(vals: np.ndarray, red: np.ndarray, axis: int, want_negative: bool) -> np.ndarray:
    """min/max under -0.0 < +0.0: where the reduced value is a zero, pick -0.0 for the min if any
    input zero is negative, +0.0 for the max if any input zero is positive."""
    is_zero = vals == 0.0
    neg = np.signbit(vals)
    if want_negative:
        has = np.any(is_zero & neg, axis=axis)
        return np.where((red == 0.0) & has, -0.0, np.where(red == 0.0, 0.0, red))
    has = np.any(is_zero & ~neg, axis=axis)
    return np.where((red == 0.0) & has, 0.0, np.where(red == 0.0, -0.0, red))


def page_summaries(keys: np.ndarray, seq_len: int, page_size: int, dtype: str):
    """Per-page, per-KV-head elementwise key min and max of one sequence.

    keys: stored keys of the sequence in logical token order, [T >= seq_len, H_kv, D].
    Returns (kmin, kmax), each [P, H_kv, D] in the storage dtype, P = ceil(seq_len / page_size);
    page p covers tokens [p*page_size, min((p+1)*page_size, seq_len)).
    """
    P = -(-seq_len // page_size)
    vals = to_f64(keys[:seq_len], dtype)
    H, D = vals.shape[1], vals.shape[2]
    kmin = np.empty((P, H, D))
    kmax = np.empty((P, H, D))
    for p in range(P):
        page = vals[p * page_size:min((p + 1) * page_size, seq_len)]
        kmin[p] = _signed_zero_fix(page, page.min(axis=0), 0, True)
        kmax[p] = _signed_zero_fix(page, page.max(axis=0), 0, False)
    return exact_to_storage(kmin, dtype), exact_to_storage(kmax, dtype)


def summary_after_append(kmin: np.ndarray, kmax: np.ndarray, k_new: np.ndarray, pos: int,
                         page_size: int, dtype: str):
    """Summary of the page that token ``pos`` lands in, after appending it (EntmaxKV
    sparse_attention_decode_paged appends k_new inside the decode call and the page
    statistics are refreshed). The first token of a page starts a fresh summary; later
    tokens widen it. kmin/kmax/k_new: [H_kv, D] stored values; returns stored values."""
    if pos % page_size == 0:
        return k_new.copy(), k_new.copy()
    old_lo, old_hi, new = to_f64(kmin, dtype), to_f64(kmax, dtype), to_f64(k_new, dtype)
    stack_lo = np.stack([old_lo, new])
    stack_hi = np.stack([old_hi, new])
    lo = _signed_zero_fix(stack_lo, stack_lo.min(axis=0), 0, True)
    hi = _signed_zero_fix(stack_hi, stack_hi.max(axis=0), 0, False)
    return exact_to_storage(lo, dtype), exact_to_storage(hi, dtype)


def page_mean_std(keys: np.ndarray, seq_len: int, page_size: int, dtype: str):
    """Per-page, per-KV-head elementwise key mean and standard deviation (EntmaxKV README,
    introduction: pages are scored from per-page key statistics, "mean/std for Gaussian";
    repository layout, gaussian/page_metadata.py, "Per-page k_mean / k_std refresh"). The
    standard deviation is the population one (divisor n, the page's valid token count); tokens
    at or past seq_len are not part of any page. keys [T >= seq_len, H_kv, D] stored. Returns
    float64 (mean, std), each [P, H_kv, D]."""
    P = -(-seq_len // page_size)
    vals = to_f64(keys[:seq_len], dtype)
    H, D = vals.shape[1], vals.shape[2]
    mean = np.empty((P, H, D))
    std = np.empty((P, H, D))
    for p in range(P):
        page = vals[p * page_size:min((p + 1) * page_size, seq_len)]
        n = page.shape[0]
        mean[p] = page.sum(axis=0) / n
        std[p] = np.sqrt(((page - mean[p]) ** 2).sum(axis=0) / n)
    return mean, std


# ----------------------------------------------------------------------------------
# S2: page score
# ----------------------------------------------------------------------------------
def quest_scores(q: np.ndarray, kmin: np.ndarray, kmax: np.ndarray, dtype: str, scale: float) -> np.ndarray:
    """Quest-style page upper bound, max over the GQA group, times ``scale``.

    q: [H_q, D] stored; kmin, kmax: [P, H_kv, D] stored. Returns float64 [H_kv, P]:
      score[h, p] = scale * max_{g in group(h)} sum_d max(q[g,d]*kmin[p,h,d], q[g,d]*kmax[p,h,d]).
    Query head g belongs to KV head g // (H_q // H_kv).
    """
    qv, lo, hi = to_f64(q, dtype), to_f64(kmin, dtype), to_f64(kmax, dtype)
    H_q = qv.shape[0]
    P, H_kv, D = lo.shape
    G = H_q // H_kv
    out = np.empty((H_kv, P))
    for h in range(H_kv):
        per_head = np.empty((G, P))
        for j in range(G):
            g = h * G + j
            per_head[j] = np.maximum(qv[g] * lo[:, h, :], qv[g] * hi[:, h, :]).sum(axis=1)
        out[h] = per_head.max(axis=0) * scale
    return out


def quest_scores_per_query_head(q: np.ndarray, kmin: np.ndarray, kmax: np.ndarray, dtype: str,
                                scale: float) -> np.ndarray:
    """The same bound for each query head on its own, with no group combine (EntmaxKV README,
    "Two selection strategies", Top-k: the pages are ranked and kept per query head).

    q: [H_q, D] stored; kmin, kmax: [P, H_kv, D] stored. Returns float64 [H_q, P]:
      score[g, p] = scale * sum_d max(q[g,d]*kmin[p,h,d], q[g,d]*kmax[p,h,d]),  h = g // (H_q // H_kv).
    """
    qv, lo, hi = to_f64(q, dtype), to_f64(kmin, dtype), to_f64(kmax, dtype)
    H_q = qv.shape[0]
    P, H_kv, D = lo.shape
    G = H_q // H_kv
    out = np.empty((H_q, P))
    for g in range(H_q):
        h = g // G
        out[g] = np.maximum(qv[g] * lo[:, h, :], qv[g] * hi[:, h, :]).sum(axis=1) * scale
    return out


def gaussian_scores(q: np.ndarray, mean: np.ndarray, std: np.ndarray, dtype: str, scale: float, z: float) -> np.ndarray:
    """Gaussian page score from the mean / std summaries (EntmaxKV README, "Two selection
    strategies", Gaussian-aware: each page's scores modelled as a Gaussian, pages kept whose
    estimated maximum is high). For query head g and page p the logits q_g . k_t of the page's
    tokens are modelled as a Gaussian with mean q_g . mean_p and variance
    sum_d q_gd^2 std_pd^2 (dimensions taken as independent); the page's estimated maximum is
    mean + z * std. Combined over the GQA group by max and scaled like the bound:

      score[h, p] = scale * max_{g in group(h)} (q_g . mean_p + z * sqrt(sum_d q_gd^2 std_pd^2)).

    q [H_q, D] stored; mean, std [P, H_kv, D] float64. Returns float64 [H_kv, P]."""
    qv = to_f64(q, dtype)
    H_q = qv.shape[0]
    P, H_kv, D = mean.shape
    G = H_q // H_kv
    out = np.empty((H_kv, P))
    for h in range(H_kv):
        per_head = np.empty((G, P))
        for j in range(G):
            g = h * G + j
            mu = mean[:, h, :] @ qv[g]
            sd = np.sqrt((std[:, h, :] ** 2) @ (qv[g] ** 2))
            per_head[j] = mu + z * sd
        out[h] = per_head.max(axis=0) * scale
    return out


# ----------------------------------------------------------------------------------
# S3: top-b selection with forced sink and tail
# ----------------------------------------------------------------------------------
def forced_pages(P: int, sink_pages: int = 1, window_pages: int = 1) -> list[int]:
    """The always-kept pages, ascending: the first ``sink_pages`` pages and the last
    ``window_pages`` pages (the tail page among them), clipped to the P pages that exist
    (LOCKS PKG-INFO, "Configuration (LocksConfig)": sink_pages / window_pages, the always-kept
    first / recent pages, default 1 / 1). With the defaults: the sink (page 0) and the tail
    (page P-1). sink_pages = 0 keeps only recent pages, as EntmaxKV's top-k does (README, "Two
    selection strategies": the budget includes the always-attended tail page)."""
    if sink_pages < 0 or window_pages < 1:
        raise ValueError("sink_pages >= 0 and window_pages >= 1 (the tail page is always kept)")
    return sorted(set(range(min(sink_pages, P))) | set(range(max(0, P - window_pages), P)))


def select_pages(scores: np.ndarray, budget: int, sink_pages: int = 1, window_pages: int = 1) -> list[int]:
    """Selected logical pages of one (sequence, KV head), ascending.

    scores: [P] page scores. The forced pages (``forced_pages``) are always kept and count
    inside the budget; the remaining min(budget, P) - |forced| pages are the highest-scoring
    others, ties going to the lower page index.
    """
    P = len(scores)
    forced = forced_pages(P, sink_pages, window_pages)
    if budget < len(forced):
        raise ValueError("budget must hold every always-kept page")
    count = min(budget, P)
    others = [p for p in range(P) if p not in forced]
    ranked = sorted(others, key=lambda p: (-float(scores[p]), p))
    return sorted(forced + ranked[:count - len(forced)])


def cutoff_score(scores: np.ndarray, budget: int, sink_pages: int = 1, window_pages: int = 1) -> float | None:
    """Score of the last non-forced page that made the cut (None if no free page is chosen by
    score: every page is kept, or the budget holds only the forced pages)."""
    P = len(scores)
    forced = forced_pages(P, sink_pages, window_pages)
    k_free = min(budget, P) - len(forced)
    if min(budget, P) >= P or k_free <= 0:
        return None
    others = [p for p in range(P) if p not in forced]
    ranked = sorted(others, key=lambda p: (-float(scores[p]), p))
    return float(scores[ranked[k_free - 1]])


# ----------------------------------------------------------------------------------
# S3 budget modes
# ----------------------------------------------------------------------------------
def retained_count(N: int, r: float) -> int:
    """Pages kept out of N for a fractional budget r: min(N, max(1, ceil(N * r))) (the
    retained-count rule of the vllm-rlt pull request #157 discussion, the commit that aligns
    the rounding with the FlashLoop reference: a ceiling, not rounding to nearest). N * r is
    evaluated in IEEE double precision, as the rule's own Python code does."""
    if N < 1:
        raise ValueError("N >= 1")
    return min(N, max(1, math.ceil(float(N) * float(r))))


def budget_for(P: int, *, fraction: float | None = None, pages: int | None = None,
               sink_pages: int = 1, window_pages: int = 1) -> int:
    """Per-(sequence, KV head) budget of a budget mode (LOCKS PKG-INFO, "Configuration
    (LocksConfig)": ``budget`` = a fixed fraction of the pages, ``budget_pages`` = a fixed
    absolute number of pages per unit). A fraction uses ``retained_count``; either mode is then
    raised to the number of always-kept pages, which the budget includes, and capped at P."""
    forced = len(forced_pages(P, sink_pages, window_pages))
    if (fraction is None) == (pages is None):
        raise ValueError("exactly one of fraction, pages")
    if fraction is not None:
        if not (0.0 < fraction <= 1.0):
            raise ValueError("fraction in (0, 1]")
        b = retained_count(P, fraction)
    else:
        if pages < 1:
            raise ValueError("pages >= 1")
        b = min(P, pages)
    return max(b, forced)


# ----------------------------------------------------------------------------------
# S3 budget mode: adaptive per-head coverage over exact page masses
# ----------------------------------------------------------------------------------
def page_masses(q: np.ndarray, keys: np.ndarray, seq_len: int, page_size: int, dtype: str, scale: float) -> np.ndarray:
    """Exact softmax mass of every page for every query head (LOCKS PKG-INFO, "Configuration
    (LocksConfig)", `coverage`: adaptive per-head nucleus coverage over exact page masses; AMASS
    PyPI page, "Key AmassConfig fields", the same option). For query head g of KV head h:

      mass[g, p] = sum over tokens t of page p (t < seq_len) of softmax_t(scale * q_g . k_{t,h}),

    the softmax taken over every token of the sequence. q [H_q, D]; keys [T >= seq_len, H_kv, D]
    stored. Returns float64 [H_q, P]; each row sums to 1."""
    qv = to_f64(q, dtype)
    H_q = qv.shape[0]
    H_kv = keys.shape[1]
    G = H_q // H_kv
    P = -(-seq_len // page_size)
    k = to_f64(keys[:seq_len], dtype)
    out = np.empty((H_q, P))
    for g in range(H_q):
        logits = scale * (k[:, g // G, :] @ qv[g])
        w = np.exp(logits - logits.max())
        w /= w.sum()
        for p in range(P):
            out[g, p] = w[p * page_size:min((p + 1) * page_size, seq_len)].sum()
    return out


def group_masses(masses: np.ndarray, H_kv: int) -> np.ndarray:
    """Page masses of each KV head: the max over the query heads of its GQA group (the group
    combine `max` of the LOCKS configuration table). [H_q, P] -> [H_kv, P]."""
    G = masses.shape[0] // H_kv
    return np.stack([masses[h * G:(h + 1) * G].max(axis=0) for h in range(H_kv)])


def select_coverage(mass: np.ndarray, coverage: float, b_max: int, sink_pages: int = 1,
                    window_pages: int = 1) -> list[int]:
    """Nucleus selection of one unit, ascending: the always-kept pages, then the other pages in
    order of (mass desc, index asc), as few as make the selected mass reach coverage times the
    unit's total mass (for a group of one query head the total is 1), and at most b_max pages in
    all (the row's capacity). mass: [P] float64."""
    P = len(mass)
    forced = forced_pages(P, sink_pages, window_pages)
    if b_max < len(forced):
        raise ValueError("b_max must hold every always-kept page")
    target = coverage * float(mass.sum())
    have = float(mass[forced].sum()) if forced else 0.0
    ranked = sorted((p for p in range(P) if p not in forced), key=lambda p: (-float(mass[p]), p))
    chosen = []
    for p in ranked:
        if have >= target or len(forced) + len(chosen) >= b_max:
            break
        chosen.append(p)
        have += float(mass[p])
    return sorted(forced + chosen)


# ----------------------------------------------------------------------------------
# S4: exact softmax attention over selected tokens
# ----------------------------------------------------------------------------------
def latent_values(keys: np.ndarray, v_head_dim: int) -> np.ndarray:
    """Values of a latent (MLA) cache: the first v_head_dim dims of each token's latent key
    (DeepSeek-shaped latent attention: one 576-dim latent per token, of which the first 512 are
    the value). keys [T, 1, D] stored -> [T, 1, v_head_dim], the same stored elements."""
    if not (0 < v_head_dim <= keys.shape[2]):
        raise ValueError("0 < v_head_dim <= head_dim")
    return keys[:, :, :v_head_dim]


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """out = softmax(scale * k q) v for one query vector; q [D], k [n, D], v [n, D_v], float64."""
    logits = scale * (k @ q)
    w = np.exp(logits - logits.max())
    return (w @ v) / w.sum()


def page_tokens(pages, seq_len: int, page_size: int) -> np.ndarray:
    """Logical token indices of the given pages, in page order, excluding tokens >= seq_len."""
    toks = [np.arange(p * page_size, min((p + 1) * page_size, seq_len)) for p in pages]
    return np.concatenate(toks) if toks else np.zeros(0, dtype=np.int64)


def attend_pages(q: np.ndarray, keys: np.ndarray, values: np.ndarray, seq_len: int, page_size: int,
                 selected, dtype: str, scale: float) -> np.ndarray:
    """Decode output of one sequence: every query head attends the tokens of its KV head's
    selected pages. q [H_q, D]; keys [T, H_kv, D]; values [T, H_kv, D_v] (logical order,
    stored); selected: per KV head a list of logical pages. Returns float64 [H_q, D_v]."""
    qv = to_f64(q, dtype)
    H_q = qv.shape[0]
    H_kv = keys.shape[1]
    G = H_q // H_kv
    out = np.empty((H_q, values.shape[2]))
    for h in range(H_kv):
        t = page_tokens(selected[h], seq_len, page_size)
        kh = to_f64(keys[t, h], dtype)
        vh = to_f64(values[t, h], dtype)
        for j in range(G):
            g = h * G + j
            out[g] = softmax_attention(qv[g], kh, vh, scale)
    return out


def attend_pages_per_query_head(q: np.ndarray, keys: np.ndarray, values: np.ndarray, seq_len: int,
                                page_size: int, selected, dtype: str, scale: float) -> np.ndarray:
    """Decode output when pages are selected per query head: query head g attends the tokens of
    its own selected pages of its KV head. selected: per query head a list of logical pages.
    Returns float64 [H_q, D_v]."""
    qv = to_f64(q, dtype)
    H_q = qv.shape[0]
    H_kv = keys.shape[1]
    G = H_q // H_kv
    out = np.empty((H_q, values.shape[2]))
    for g in range(H_q):
        h = g // G
        t = page_tokens(selected[g], seq_len, page_size)
        out[g] = softmax_attention(qv[g], to_f64(keys[t, h], dtype), to_f64(values[t, h], dtype), scale)
    return out


def dense_attention(q, keys, values, seq_len, page_size, dtype, scale):
    """Full-KV decode of one sequence (every page of every KV head)."""
    P = -(-seq_len // page_size)
    H_kv = keys.shape[1]
    return attend_pages(q, keys, values, seq_len, page_size, [list(range(P))] * H_kv, dtype, scale)


# ----------------------------------------------------------------------------------
# paged-cache views (the vLLM layout [num_blocks, page_size, H_kv, D] per K / V)
# ----------------------------------------------------------------------------------
def logical_from_cache(cache: np.ndarray, block_row: np.ndarray, seq_len: int, page_size: int) -> np.ndarray:
    """Gather one sequence's tokens [seq_len, H, Dc] out of a paged cache through its block-table row."""
    P = -(-seq_len // page_size)
    pages = [cache[int(block_row[p])] for p in range(P)]
    return np.concatenate(pages, axis=0)[:seq_len]


# ----------------------------------------------------------------------------------
# one decode step of one sequence, end to end
# ----------------------------------------------------------------------------------
def decode_step(q, keys, values, seq_len, page_size, budget, dtype, scale, sink_pages=1, window_pages=1):
    """Score, select and attend for one sequence whose keys/values (logical order) already
    include the current token. Returns (summaries (kmin, kmax), scores [H_kv, P],
    selected per KV head, out [H_q, D_v])."""
    kmin, kmax = page_summaries(keys, seq_len, page_size, dtype)
    scores = quest_scores(q, kmin, kmax, dtype, scale)
    selected = [select_pages(scores[h], budget, sink_pages, window_pages) for h in range(scores.shape[0])]
    out = attend_pages(q, keys, values, seq_len, page_size, selected, dtype, scale)
    return (kmin, kmax), scores, selected, out


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
