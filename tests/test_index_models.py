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
