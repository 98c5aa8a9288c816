"""Executable models of two pieces of kernel index logic, checked on the CPU (no GPU, no oracle).

1. The score kernel's 1-D grid: CTAs of the body region (chunks of pchunk pages of each
   sequence's first P - T pages) followed by CTAs of the tail region (each sequence's last T
   pages in chunks of tail_chunk), decoded from the block index the way page_score_kernel does,
   with T and the chunk counts sized the way its launcher does. Every (head group, sequence,
   page) must be scored exactly once, for any lengths, including bad ones (skipped) and T
   clamped to max_pages.
2. The selection kernel's radix select: MSB-first 8-bit digits from the highest bit where the
   smallest and largest nonzero keys differ, stopping early when the chosen bin holds exactly the
   keys still needed, then the "key > T, plus the first need_eq keys equal to T" compaction. The
   chosen set must equal the top k by (key desc, index asc), ties included.
3. The latent decode's split plan and its cluster merge: the planner's split width (waves of one
   CTA per SM against the merge's cost) must cover every list entry once with at most 128 splits;
   with at most 8 splits per (sequence, half) the merge runs in a cluster, where rank r writes the
   value dims [r·span, (r+1)·span) of every head through four warps that take head pairs
   warp + 4u + 16j and, per half-warp, 4-dim pieces 64 apart. Every (head, value dim) of the half
   must be written exactly once, and no remote rank at or past the cluster size is addressed.
"""
import random


# ------------------------------------------------------------------ 1. score grid
def _score_launch(B, n_grp, max_pages, pchunk, slots, tail_chunk, waves=1, tail_override=None):
    rows = B * n_grp
    tail = -(-slots * tail_chunk * waves // rows) if tail_override is None else tail_override
    tail = -(-tail // tail_chunk) * tail_chunk
    tail_pages = max(0, min(tail, max_pages))
    return dict(tail_pages=tail_pages, tail_chunk=tail_chunk, tail_chunks=-(-tail_pages // tail_chunk),
                body_chunks=-(-max_pages // pchunk), pchunk=pchunk)


def _score_cta_pages(a, B, n_grp, bx, lens_pages, max_pages):
    """Pages (group, sequence, page) CTA bx scores, or [] when it leaves at once."""
    n_body = a["body_chunks"] * B * n_grp
    x = bx
    in_tail = x >= n_body
    if in_tail:
        x -= n_body
    per = a["tail_chunks"] if in_tail else a["body_chunks"]
    c, x = x % per, x // per
    i, g = x % B, x // B
    P = lens_pages[i]
    if P < 1 or P > max_pages:
        return []
    body_end = P - min(P, a["tail_pages"])
    p0 = body_end + c * a["tail_chunk"] if in_tail else c * a["pchunk"]
    p1 = min(P, p0 + a["tail_chunk"]) if in_tail else min(body_end, p0 + a["pchunk"])
    return [(g, i, p) for p in range(p0, p1)]


def test_score_grid_covers_every_page_once():
    rng = random.Random(5)
    for _ in range(400):
        B, n_grp, mp = rng.randint(1, 70), rng.choice([1, 2]), rng.randint(1, 600)
        lens = [rng.choice([0, rng.randint(1, mp), mp, mp + 1]) for _ in range(B)]
        a = _score_launch(B, n_grp, mp, rng.choice([16, 32, 64]), 608, rng.choice([1, 8, 16, 24]),
                          tail_override=rng.choice([None, None, 0, 5, 10000]))
        n_ctas = (a["body_chunks"] + a["tail_chunks"]) * B * n_grp
        seen = {}
        for bx in range(n_ctas):
            for key in _score_cta_pages(a, B, n_grp, bx, lens, mp):
                assert key not in seen
                seen[key] = bx
        want = {(g, i, p) for i in range(B) if 1 <= lens[i] <= mp for g in range(n_grp) for p in range(lens[i])}
        assert set(seen) == want


# ------------------------------------------------------------------ 2. radix select
def _radix_select(keys, k, early_exit):
    nz = [x for x in keys if x]
    kmin, kmax = min(nz), max(nz)
    diff = kmin ^ kmax
    top = diff.bit_length() - 1 if diff else 0
    shift = top - 7 if top >= 7 else 0
    prefix = 0 if shift + 8 >= 32 else (kmin >> (shift + 8)) << (shift + 8)
    mask = 0 if shift + 8 >= 32 else (0xFFFFFFFF << (shift + 8)) & 0xFFFFFFFF
    need = k
    while True:
        hist = [0] * 256
        for x in keys:
            if x and (x & mask) == prefix:
                hist[(x >> shift) & 255] += 1
        incl = 0
        for d in range(255, -1, -1):
            excl, incl = incl, incl + hist[d]
            if excl < need <= incl:
                break
        need -= excl
        prefix |= d << shift
        mask |= 255 << shift
        if shift == 0:
            break
        if early_exit and hist[d] == need:
            return (prefix - 1 if prefix else 0), 0
        shift = shift - 8 if shift >= 8 else 0
    return prefix, need


def _compact(keys, T, need_eq):
    out, seen = [], 0
    for i, x in enumerate(keys):
        if x > T:
            out.append(i)
        elif x == T and x != 0:
            if seen < need_eq:
                out.append(i)
            seen += 1
    return out


def test_radix_select_with_early_exit_is_the_top_k():
    rng = random.Random(7)
    for _ in range(3000):
        n = rng.randint(2, 400)
        kind = rng.random()
        if kind < 0.3:
            keys = [rng.randint(1, 2 ** 32 - 1) for _ in range(n)]
        elif kind < 0.6:
            keys = [rng.randint(1, 20) for _ in range(n)]  # heavy ties
        else:
            keys = [rng.choice([0, rng.randint(1 << 31, (1 << 31) + 1000)]) for _ in range(n)]
        nz = sum(1 for x in keys if x)
        if nz <= 1:
            continue
        k = rng.randint(1, nz - 1)
        ref = sorted((i for i, x in enumerate(keys) if x), key=lambda i: (-keys[i], i))[:k]
        for early in (False, True):
            T, need_eq = _radix_select(keys, k, early)
            assert sorted(_compact(keys, T, need_eq)) == sorted(ref)


# ------------------------------------------------------------------ 3. latent split plan and merge
_MLA_MAX_SW, _MLA_MAX_ITEMS, _MLA_CLUSTER_MAX = 128, 128, 8


def _mla_plan(units, entries, sms=152):
    """Split width and count the way the latent decode's planner picks them."""
    e = max(entries, 1)
    sw, best = max(1, min(entries, _MLA_MAX_SW)), 1e300
    for items in range(1, min(e, _MLA_MAX_ITEMS) + 1):
        w = -(-e // items)
        if w > _MLA_MAX_SW:
            continue
        n = -(-e // w)
        waves = -(-(units * n) // sms)
        cost = waves * (w + 2.0) + (1.0 if n <= _MLA_CLUSTER_MAX else 1.0 * n)
        if cost < best - 1e-9:
            best, sw = cost, w
    return sw, -(-entries // sw)


def _cluster_merge_writes(n, rank, m_of_rank):
    """(head, dim) pairs CTA `rank` of an n-CTA cluster writes, and the ranks whose rows it reads:
    rank k's row is read only where its merge weight is nonzero, and the weight of every k at or
    past the cluster size, or of a split with no tiles (m = -inf), is 0."""
    span = (-(-256 // n) + 3) & ~3
    d0 = min(256, rank * span)
    d1 = min(256, d0 + span)
    mk = [m_of_rank[k] if k < n else float("-inf") for k in range(_MLA_CLUSTER_MAX)]
    weight_nonzero = [m != float("-inf") for m in mk]
    writes, ranks = [], set()
    for warp in range(4):
        for lane in range(32):
            hl, l16 = lane >> 4, lane & 15
            for pb in range(warp, 64, 16):
                d = d0 + l16 * 4
                while d < d1:
                    for u in range(4):
                        h = 2 * (pb + 4 * u) + hl
                        ranks.update(k for k in range(_MLA_CLUSTER_MAX) if weight_nonzero[k])
                        writes.extend((h, d + j) for j in range(4) if d + j < d1)
                    d += 64
    return writes, ranks


def test_latent_split_plan_covers_every_entry():
    rng = random.Random(7)
    cases = [(32, 103), (2, 103), (8, 103), (160, 3), (4, 3), (4, 7), (6, 16), (32, 2048), (2, 1)]
    cases += [(rng.randint(1, 400), rng.randint(1, 4096)) for _ in range(300)]
    for units, entries in cases:
        sw, n = _mla_plan(units, entries)
        assert 1 <= sw <= _MLA_MAX_SW and n <= _MLA_MAX_ITEMS
        covered = [e for s in range(n) for e in range(s * sw, min(entries, (s + 1) * sw))]
        assert covered == list(range(entries))
    assert _mla_plan(32, 103) == (26, 4)       # the latent workload: clusters of 4 splits
    assert _mla_plan(160, 3)[1] == 1            # more units than SMs: one split each
    assert _mla_plan(4, 3)[1] == 3 and _mla_plan(4, 7)[1] == 7


def test_cluster_merge_writes_every_value_dim_once():
    rng = random.Random(3)
    for n in range(1, _MLA_CLUSTER_MAX + 1):
        # some splits of a short list have no tiles (m = -inf); at least one has
        m = [rng.choice([float("-inf"), rng.uniform(-4.0, 4.0)]) for _ in range(n)]
        m[rng.randrange(n)] = 0.5
        seen = {}
        for r in range(n):
            writes, ranks = _cluster_merge_writes(n, r, m)
            assert ranks == {k for k in range(n) if m[k] != float("-inf")} and ranks <= set(range(n))
            for key in writes:
                assert key not in seen, (n, r, key)
                seen[key] = r
        assert set(seen) == {(h, d) for h in range(128) for d in range(256)}, n
