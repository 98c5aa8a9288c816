"""The allocation-free sparse decode entry point.

psk_sparse_paged_decode_noalloc serves callers that may not allocate device memory (hosts that
own all device memory and pass a plugin only inputs and outputs, or loops that must never call
cudaMalloc). It keeps its split partials in a fixed per-device array inside the library instead
of a caller workspace. These tests call it through the C ABI and check it against the workspace
entry point, twice in a row (the array keeps the previous call's contents), and check that a
problem too large for the fixed array is refused. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

from parity import check_output

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import page_sparse_kv_gb300 as psk  # noqa: E402
from workloads.device import budgets as dev_budgets, from_torch, to_torch, upload  # noqa: E402


@pytest.fixture(scope="module")
def cache_and_workload():
    from page_sparse_kv_gb300.build import build
    build()
    w = W.reduced(3)
    return upload(w), w


def test_noalloc_matches_workspace_decode_twice(cache_and_workload):
    cache, w = cache_and_workload
    L = cache.layout
    for step in (0, 1):
        q = to_torch(w.queries(step), w.dtype).cuda()
        sel = cache.score_select(q, dev_budgets(w))
        ref = cache.sparse_decode(q, sel)
        got = torch.full_like(ref, float("nan"))
        psk.sparse_paged_decode_noalloc(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, sel,
                                        cache.b_max, cache.scale, got)
        torch.cuda.synchronize()
        g = from_torch(got.float(), "f32")
        r = from_torch(ref.float(), "f32").astype(np.float64)
        assert np.all(np.isfinite(g))
        check_output(g, r, w.dtype)


def test_noalloc_refuses_problems_beyond_its_scratch(cache_and_workload):
    """The refusal happens on the host, before any launch. The layout is first checked, by the
    host-only size query, to need more than the fixed array; only then is the entry point called
    (its pointer arguments are placeholders that no kernel may ever see)."""
    big = psk.Layout(4096, 32, 8, 128, 128, 16, 1 << 20, 8192)
    need = psk.sparse_decode_workspace_size(big, 8192)
    if not need > (32 << 20):
        pytest.fail(f"layout needs only {need} bytes of scratch: it would be accepted, so it is not called")
    P = ctypes.c_void_p
    rc = psk.lib().psk_sparse_paged_decode_noalloc(ctypes.byref(big.c()), P(256), P(256), P(256), P(256), P(256),
                                                   P(256), 8192, 0.1, P(256), None)
    assert rc == 3  # PSK_ERR_WORKSPACE: the partials would not fit the fixed array
