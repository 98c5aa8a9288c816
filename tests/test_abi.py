"""The C-ABI library builds, loads and exports every symbol include/psk.h declares; host-side
argument checks answer without a GPU (no kernel is launched by any call here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from page_sparse_kv_gb300.build import build
    build()
    import page_sparse_kv_gb300 as psk
    return psk.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "psk.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(psk_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    import page_sparse_kv_gb300 as psk
    assert set(psk.EXPORTS) == set(names)


def test_status_strings_and_version(lib):
    import page_sparse_kv_gb300 as psk
    assert psk.version() == 100
    for code in range(5):
        assert lib.psk_status_string(code)
    assert lib.psk_status_string(99) == b"unknown status"


def test_host_checks_reject_before_launch(lib):
    import page_sparse_kv_gb300 as psk
    good = psk.Layout(2, 32, 8, 128, 128, 16, 100, 50)
    assert psk.score_select_workspace_size(good, 10) > 256
    assert psk.sparse_decode_workspace_size(good, 10) > 256
    assert psk.dense_decode_workspace_size(good) > 256
    assert psk.append_workspace_size(good) == 256
    # unsupported head dim / group size / page size -> size 0
    assert psk.score_select_workspace_size(psk.Layout(2, 32, 8, 96, 96, 16, 100, 50), 10) == 0
    assert psk.dense_decode_workspace_size(psk.Layout(2, 24, 8, 128, 128, 16, 100, 50)) == 0
    assert psk.dense_decode_workspace_size(psk.Layout(2, 32, 8, 128, 128, 8, 100, 50)) == 0
    # G = 8 is built for bf16 at head_dim 128 only (tensor-core score and decode)
    assert psk.score_select_workspace_size(psk.Layout(2, 64, 8, 128, 128, 16, 100, 50), 10) > 256
    assert psk.sparse_decode_workspace_size(psk.Layout(2, 64, 8, 128, 128, 16, 100, 50), 10) > 256
    assert psk.score_select_workspace_size(psk.Layout(2, 64, 8, 64, 64, 16, 100, 50), 10) == 0
    assert psk.score_select_workspace_size(psk.Layout(2, 64, 8, 128, 128, 16, 100, 50, psk.PSK_F32), 10) == 0
    # invalid layouts
    assert psk.append_workspace_size(psk.Layout(0, 32, 8, 128, 128, 16, 100, 50)) == 0
    assert psk.append_workspace_size(psk.Layout(1, 30, 8, 128, 128, 16, 100, 50)) == 0
    L = good.c()
    P = ctypes.c_void_p
    # null pointers -> PSK_ERR_INVALID_ARG without touching the GPU
    rc = lib.psk_page_score_select(ctypes.byref(L), None, None, None, None, None, 10, 1.0, None, None, None, 0, None)
    assert rc == 1
    rc = lib.psk_dense_paged_decode(ctypes.byref(L), None, None, None, None, None, 1.0, None, None, 0, None)
    assert rc == 1
    rc = lib.psk_sparse_paged_decode(ctypes.byref(L), P(16), P(16), P(16), P(16), P(16), None, 10, 1.0, P(16),
                                     P(16), 1 << 30, None)
    assert rc == 1
    # misaligned pointer
    rc = lib.psk_dense_paged_decode(ctypes.byref(L), P(17), P(16), P(16), P(16), P(16), 1.0, P(16), P(16), 1 << 30,
                                    None)
    assert rc == 1
    # too-small workspace -> PSK_ERR_WORKSPACE
    rc = lib.psk_dense_paged_decode(ctypes.byref(L), P(16), P(16), P(16), P(16), P(16), 1.0, P(16), P(16), 64, None)
    assert rc == 3
    # empty append is a no-op that returns OK before any launch
    rc = lib.psk_kv_append_and_summarize(ctypes.byref(L), None, None, P(16), P(16), 0, 0, P(16), P(16), P(16), P(16),
                                         P(16), 256, None)
    assert rc == 0
    # the bounded-wait self-test: no workspace, a small one, or a poll limit outside 1 .. 2^22
    assert lib.psk_selftest_bounded_wait(None, 256, 10, None) == 1
    assert lib.psk_selftest_bounded_wait(P(256), 64, 10, None) == 3
    assert lib.psk_selftest_bounded_wait(P(256), 256, 0, None) == 1
    assert lib.psk_selftest_bounded_wait(P(256), 256, (1 << 22) + 1, None) == 1


def test_select_params_host_checks(lib):
    """The general score/select entry rejects bad always-kept sizes, budget modes and a b_max
    too small for a scalar budget mode before any launch (the workspace is too small here, so a
    call that got past the checks would answer PSK_ERR_WORKSPACE, still without a launch)."""
    import page_sparse_kv_gb300 as psk
    L = psk.Layout(2, 32, 8, 128, 128, 16, 100, 50).c()
    P = ctypes.c_void_p

    def call(b_max, **kw):
        prm = psk.PskSelectParams()
        prm.budgets = kw.get("budgets")
        prm.budget_fraction = kw.get("fraction", 0.0)
        prm.budget_pages = kw.get("pages", 0)
        prm.mode = kw.get("mode", psk.BUDGET_PER_SEQUENCE)
        prm.sink_pages = kw.get("sink", 1)
        prm.window_pages = kw.get("window", 1)
        prm.per_query_head = kw.get("pqh", 0)
        return lib.psk_page_score_select_ex(ctypes.byref(L), P(16), P(16), P(16), P(16), ctypes.byref(prm), b_max,
                                            1.0, P(16), None, P(16), 64, None)

    assert call(10, budgets=16) == 3                                          # checks pass, workspace short
    assert call(10) == 1                                                      # per-sequence without budgets
    assert call(10, budgets=16, sink=-1) == 1 and call(10, budgets=16, window=0) == 1
    assert call(10, budgets=16, sink=0) == 3                                  # recent pages only
    assert call(10, budgets=16, pqh=1) == 3 and call(10, budgets=16, pqh=2) == 1
    assert call(10, mode=7, budgets=16) == 1
    assert call(10, mode=psk.BUDGET_PAGES, pages=0) == 1
    assert call(10, mode=psk.BUDGET_PAGES, pages=10) == 3
    assert call(10, mode=psk.BUDGET_PAGES, pages=11) == 1                     # 11 pages exceed b_max
    assert call(12, mode=psk.BUDGET_PAGES, pages=4, sink=4, window=8) == 3   # raised to the 12 kept
    assert call(11, mode=psk.BUDGET_PAGES, pages=4, sink=4, window=8) == 1
    assert call(10, mode=psk.BUDGET_FRACTION, fraction=0.0) == 1
    assert call(10, mode=psk.BUDGET_FRACTION, fraction=1.5) == 1
    assert call(3, mode=psk.BUDGET_FRACTION, fraction=0.05) == 3             # ceil(50 * 0.05) = 3
    assert call(2, mode=psk.BUDGET_FRACTION, fraction=0.05) == 1
    assert call(49, mode=psk.BUDGET_FRACTION, fraction=1.0) == 1             # every one of 50 pages
    # the decode with flags: unknown flag bits, or no selected rows, answer before any launch
    # (0x4 is no flag; every call here must be refused before a launch, since its pointers are
    # placeholders)
    rc = lib.psk_sparse_paged_decode_ex(ctypes.byref(L), P(16), P(16), P(16), P(16), P(16), P(16), 10, 1.0, 0x4,
                                        P(16), P(16), 1 << 30, None)
    assert rc == 1
    # the host value tier is refused for shapes it is not built for (fp32 here)
    L32 = psk.Layout(2, 32, 8, 128, 128, 16, 100, 50, dtype=psk.PSK_F32).c()
    rc = lib.psk_sparse_paged_decode_ex(ctypes.byref(L32), P(16), P(16), P(16), P(16), P(16), P(16), 10, 1.0, 0x2,
                                        P(16), P(16), 1 << 30, None)
    assert rc == 2
    rc = lib.psk_sparse_paged_decode_ex(ctypes.byref(L), P(16), P(16), P(16), P(16), P(16), None, 10, 1.0, 0x1,
                                        P(16), P(16), 1 << 30, None)
    assert rc == 1
    rc = lib.psk_sparse_paged_decode_ex(ctypes.byref(L), P(16), P(16), P(16), P(16), P(16), P(16), 10, 1.0, 0x1,
                                        P(16), P(16), 64, None)
    assert rc == 3
    # one workspace covers the per-query-head form too
    big = psk.Layout(2, 32, 8, 128, 128, 16, 100, 50)
    assert psk.score_select_workspace_size(big, 10) > 0 and psk.sparse_decode_workspace_size(big, 10) > 0


def test_workspace_sizes_cover_every_form(lib):
    """Host planning only: for a spread of layouts each call's workspace size is positive, the
    combined size covers all of them, and a GQA layout's score / decode sizes also cover its
    per-query-head form (one workspace serves both)."""
    import page_sparse_kv_gb300 as psk
    cases = [  # batch, H_q, H_kv, D, page, num_blocks, max_pages, dtype
        (64, 32, 8, 128, 16, 150000, 4096, psk.PSK_BF16),
        (1, 32, 8, 128, 16, 70000, 65536, psk.PSK_BF16),
        (3, 16, 8, 64, 32, 500, 200, psk.PSK_BF16),
        (5, 8, 8, 128, 64, 900, 300, psk.PSK_BF16),
        (2, 4, 1, 64, 16, 300, 100, psk.PSK_F32),
        (7, 64, 16, 128, 48, 2000, 333, psk.PSK_BF16),
    ]
    for B, Hq, Hkv, D, ps, nb, mp, dt in cases:
        L = psk.Layout(B, Hq, Hkv, D, D, ps, nb, mp, dtype=dt)
        V = psk.Layout(B, Hq, Hq, D, D, ps, nb, mp, dtype=dt)  # the per-query-head view's shape
        for b in (2, 5, 128, min(mp, 2048)):
            sizes = [psk.append_workspace_size(L), psk.score_select_workspace_size(L, b),
                     psk.sparse_decode_workspace_size(L, b), psk.dense_decode_workspace_size(L)]
            assert min(sizes) > 0, (L, b, sizes)
            assert psk.workspace_size(L, b) == max(sizes)
            assert psk.score_select_workspace_size(L, b) >= psk.score_select_workspace_size(V, b)
            assert psk.sparse_decode_workspace_size(L, b) >= psk.sparse_decode_workspace_size(V, b)
    # the selection limit: 65536 pages allow b_max 2049 (4 chunks of 16384 x 2048 winners = 8192),
    # not 2050
    L = psk.Layout(1, 32, 8, 128, 128, 16, 70000, 65536)
    assert psk.score_select_workspace_size(L, 2049) > 0 and psk.score_select_workspace_size(L, 2050) == 0
    # the latent form has its own sizes and no per-query-head form
    M = psk.Layout(16, 128, 1, 576, 512, 64, 40000, 2048, latent=1)
    assert psk.score_select_workspace_size(M, 103) > 0 and psk.sparse_decode_workspace_size(M, 103) > 0


def test_score_select_launch_count(lib):
    """Two launches for GQA caches (score, selection), three for the latent form."""
    import page_sparse_kv_gb300 as psk
    batched = psk.Layout(64, 32, 8, 128, 128, 16, 150000, 4096)
    assert psk.score_select_launches(batched, 205) == 2
    assert psk.score_select_launches(batched, 205, per_query_head=True) == 2
    long_ctx = psk.Layout(1, 32, 8, 128, 128, 16, 65536, 65536)
    assert psk.score_select_launches(long_ctx, 128) == 2
    latent = psk.Layout(16, 128, 1, 576, 512, 64, 40000, 2048, psk.PSK_BF16, 1)
    assert psk.score_select_launches(latent, 103) == 3
    assert psk.score_select_launches(psk.Layout(2, 32, 8, 96, 96, 16, 100, 50), 10) == 0


def test_new_entry_points_reject_before_launch(lib):
    """Coverage, mean/std append, Gaussian score and the value tier: host checks answer without a
    GPU (every call here is refused before any launch)."""
    import page_sparse_kv_gb300 as psk
    P = ctypes.c_void_p
    L = psk.Layout(2, 32, 8, 128, 128, 16, 100, 50).c()
    latent = psk.Layout(2, 128, 1, 576, 512, 64, 100, 50, psk.PSK_BF16, 1).c()
    f32 = psk.Layout(2, 4, 1, 64, 64, 16, 100, 50, psk.PSK_F32).c()
    big = 1 << 30
    # coverage: sizes, null pointers, coverage outside (0, 1], latent, small workspace
    assert psk.coverage_workspace_size(psk.Layout(2, 32, 8, 128, 128, 16, 100, 50), 10) > \
        psk.score_select_workspace_size(psk.Layout(2, 32, 8, 128, 128, 16, 100, 50), 10)
    assert lib.psk_coverage_workspace_size(ctypes.byref(latent), 10) == 0
    cov = lib.psk_page_select_coverage
    assert cov(ctypes.byref(L), None, P(16), P(16), P(16), 0.9, 1, 1, 10, 1.0, P(16), None, P(16), big, None) == 1
    assert cov(ctypes.byref(L), P(16), P(16), P(16), P(16), 0.0, 1, 1, 10, 1.0, P(16), None, P(16), big, None) == 1
    assert cov(ctypes.byref(L), P(16), P(16), P(16), P(16), 1.5, 1, 1, 10, 1.0, P(16), None, P(16), big, None) == 1
    assert cov(ctypes.byref(L), P(16), P(16), P(16), P(16), 0.9, 1, 0, 10, 1.0, P(16), None, P(16), big, None) == 1
    assert cov(ctypes.byref(latent), P(16), P(16), P(16), P(16), 0.9, 1, 1, 10, 1.0, P(16), None, P(16), big,
               None) == 2
    assert cov(ctypes.byref(L), P(16), P(16), P(16), P(16), 0.9, 1, 1, 10, 1.0, P(16), None, P(16), 64, None) == 3
    # append with the mean / std store: one store at least, 16-byte aligned
    ap = lib.psk_kv_append_and_summarize_ex
    assert ap(ctypes.byref(L), P(16), P(16), P(16), P(16), 1, 1, P(16), P(16), None, None, P(16), P(16), 256,
              None) == 1
    assert ap(ctypes.byref(L), P(16), P(16), P(16), P(16), 1, 1, P(16), P(16), None, P(20), P(16), P(16), 256,
              None) == 1
    assert ap(ctypes.byref(L), P(16), P(16), P(16), P(16), 0, 0, P(16), P(16), None, P(16), P(16), P(16), 256,
              None) == 0  # nothing to append: OK before any launch
    # Gaussian score: stats required; per-query-head rows and latent caches are not built
    prm = psk.select_params(budgets=torch_free_budgets())
    g = lib.psk_page_score_select_gaussian
    assert g(ctypes.byref(L), P(16), None, P(16), P(16), ctypes.byref(prm), 10, 1.0, 1.5, P(16), None, P(16), big,
             None) == 1
    assert g(ctypes.byref(L), P(16), P(16), P(16), P(16), ctypes.byref(prm), 10, 1.0, float("nan"), P(16), None,
             P(16), big, None) == 1
    prm_q = psk.select_params(budgets=torch_free_budgets(), per_query_head=True)
    assert g(ctypes.byref(L), P(16), P(16), P(16), P(16), ctypes.byref(prm_q), 10, 1.0, 1.5, P(16), None, P(16),
             big, None) == 2
    # value tier: hot buffer and slot map required; fill only for bf16 GQA with head_dim 128
    t = lib.psk_sparse_paged_decode_tiered
    assert t(ctypes.byref(L), P(16), P(16), P(16), P(16), 0, P(16), P(16), P(16), P(16), 10, 1.0, P(16), P(16), big,
             None) == 1
    assert t(ctypes.byref(L), P(16), P(16), P(16), P(16), 4, None, P(16), P(16), P(16), 10, 1.0, P(16), P(16), big,
             None) == 1
    fill = lib.psk_value_tier_fill
    assert fill(ctypes.byref(latent), P(16), P(16), P(16), 1, P(16), 4, P(16), P(16), 256, None) == 2
    assert fill(ctypes.byref(f32), P(16), P(16), P(16), 1, P(16), 4, P(16), P(16), 256, None) == 2
    assert fill(ctypes.byref(L), P(16), P(16), None, 1, P(16), 4, P(16), P(16), 256, None) == 1
    assert fill(ctypes.byref(L), P(16), P(16), P(16), -1, P(16), 4, P(16), P(16), 256, None) == 1
    assert fill(ctypes.byref(L), P(16), P(16), P(16), 0, P(16), 4, P(16), P(16), 256, None) == 0  # nothing to do


def torch_free_budgets():
    """A stand-in for a device budget tensor: select_params only needs its pointer."""
    class _T:
        is_cuda = True

        def is_pinned(self):
            return False

        def is_contiguous(self):
            return True

        def data_ptr(self):
            return 16
    return _T()
