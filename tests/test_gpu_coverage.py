"""GPU parity of the adaptive coverage selection (psk_page_select_coverage) against the oracle.

The page masses (fp32 on the GPU) are checked against oracle.page_masses / group_masses; the
selected rows must be a valid nucleus under the oracle's masses (parity.compare_coverage:
identical to oracle.select_coverage except where fp32 rounding of the masses can move a page
across the boundary); and the sparse decode over the GPU's rows matches the oracle's attention
over the same pages. Cases span several selection chunks, ragged tails, every group size, both
dtypes, sink / window sets, b_max caps and coverages from a few percent to one.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from parity import MASS_REL, check_output, compare_coverage

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import page_sparse_kv_gb300 as psk  # noqa: E402
from workloads.device import from_torch, to_torch, upload  # noqa: E402

DIFFERENT = {"rows": 0, "differ": 0}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from page_sparse_kv_gb300.build import build
    build()
    yield
    print(f"coverage rows compared: {DIFFERENT['rows']}, differing from the oracle's within the fp32 band: "
          f"{DIFFERENT['differ']}")


def _custom(seq_lens, ps=16, dtype="bf16", H_q=8, H_kv=2, D=128, n_hot=4, seed=21):
    return W.Workload("coverage", seed, dtype, B=len(seq_lens), H_q=H_q, H_kv=H_kv, D=D, D_v=D, page_size=ps,
                      seq_lens=seq_lens, budgets=[2] * len(seq_lens), n_hot=n_hot, hot_rule="random", pool_slack=3)


def _run(w, coverage, b_max, S=1, Wn=1, q_scale=1.0):
    cache = upload(w)
    L = cache.layout
    q_np = w.queries()
    if q_scale != 1.0:  # sharper attention: larger logits
        q_np = W.f32_to_bf16_bits(O.to_f64(q_np, w.dtype).astype(np.float32) * np.float32(q_scale)) \
            if w.dtype == "bf16" else (q_np * np.float32(q_scale)).astype(np.float32)
    q = to_torch(q_np, w.dtype).cuda()
    ws = psk.make_workspace(L, b_max, coverage=True)
    sel = torch.full((w.B, w.H_kv, b_max), -7, dtype=torch.int32, device="cuda")
    masses = torch.full((w.B, w.H_kv, w.max_pages), float("nan"), device="cuda")
    psk.page_select_coverage(L, q, cache.k_cache, cache.block_table, cache.seq_lens, coverage, b_max, cache.scale, sel,
                             ws, sink_pages=S, window_pages=Wn, masses_out=masses)
    out = torch.empty(w.B, w.H_q, w.D_v, dtype=cache.dtype, device="cuda")
    psk.sparse_paged_decode(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, sel, b_max,
                            cache.scale, out, ws)
    torch.cuda.synchronize()
    assert psk.get_device_status(ws) == 0
    sel_np, m_np = sel.cpu().numpy(), masses.cpu().numpy()
    out_np = from_torch(out.float(), "f32")
    scale = 1.0 / math.sqrt(w.D)
    for i in range(w.B):
        n = int(w.seq_lens[i])
        P = -(-n // w.page_size)
        keys, vals = w.keys(i), w.values(i)
        gm = O.group_masses(O.page_masses(q_np[i], keys, n, w.page_size, w.dtype, scale), w.H_kv)
        for h in range(w.H_kv):
            err = np.abs(m_np[i, h, :P] - gm[h]).max()
            assert err <= MASS_REL * gm[h].max(), f"seq {i} head {h}: mass err {err:.3e}"
        use = []
        for h in range(w.H_kv):
            ok, same, got, ref = compare_coverage(sel_np[i, h], gm[h], coverage, b_max, S, Wn)
            assert ok, f"seq {i} head {h}: selected {got} vs oracle {ref}"
            DIFFERENT["rows"] += 1
            DIFFERENT["differ"] += not same
            use.append(got)
        check_output(out_np[i], O.attend_pages(q_np[i], keys, vals, n, w.page_size, use, w.dtype, scale), w.dtype)
    return sel_np


@pytest.mark.parametrize("case", [
    dict(seq_lens=[16 * 300 + 5, 16 * 77, 16 * 40 + 9, 33, 1], coverage=0.95, b_max=64),
    dict(seq_lens=[16 * 300 + 5, 16 * 77, 16 * 40 + 9], coverage=0.5, b_max=300, q_scale=4.0),
    dict(seq_lens=[16 * 300 + 5, 16 * 77], coverage=1.0, b_max=400),
    dict(seq_lens=[16 * 300 + 5, 16 * 77], coverage=0.05, b_max=20, S=0, Wn=3),
    dict(seq_lens=[16 * 120 + 7, 16 * 50], coverage=0.9, b_max=16, S=2, Wn=2, q_scale=3.0),   # b_max cap
    dict(seq_lens=[16 * 90 + 3, 300], coverage=0.8, b_max=60, dtype="f32", D=64, H_q=4, H_kv=1),
    dict(seq_lens=[16 * 90 + 3, 300], coverage=0.8, b_max=60, dtype="f32", D=128, H_q=2, H_kv=2),
    dict(seq_lens=[16 * 70 + 3, 500], coverage=0.9, b_max=80, D=64, H_q=8, H_kv=4),
    dict(seq_lens=[16 * 45 + 8, 300], coverage=0.7, b_max=50, H_q=16, H_kv=8, q_scale=2.0),
    dict(seq_lens=[64 * 40 + 33, 64 * 9], coverage=0.9, b_max=30, ps=64),
])
def test_coverage_selection_parity(case):
    extra = {k: case[k] for k in ("ps", "dtype", "D", "H_q", "H_kv") if k in case}
    w = _custom(case["seq_lens"], **extra)
    _run(w, case["coverage"], case["b_max"], case.get("S", 1), case.get("Wn", 1), case.get("q_scale", 1.0))


def test_coverage_chunked_selection_long_sequence():
    """A sequence of 20,000 pages: the selection runs chunk by chunk with a merge."""
    w = _custom([16 * 20000 - 3, 16 * 5000], dtype="f32", D=64, H_q=4, H_kv=1, n_hot=8)
    _run(w, 0.3, 600, q_scale=3.0)


def test_coverage_reduces_to_plain_selection_of_every_page():
    """coverage = 1 with a b_max above every page count keeps every page; the output then equals
    the dense decode."""
    w = _custom([16 * 60 + 5, 16 * 20])
    sel = _run(w, 1.0, 128)
    for i in range(w.B):
        P = -(-int(w.seq_lens[i]) // w.page_size)
        for h in range(w.H_kv):
            assert [int(x) for x in sel[i, h] if x >= 0] == list(range(P))
