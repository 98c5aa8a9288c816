"""Python binding of libpsk, the C ABI of page-selective sparse paged decode attention.

Argument marshalling only: every step runs in the library's CUDA kernels. Tensors are
torch CUDA tensors (torch provides device memory and streams); each call passes their
device pointers, the layout and the current torch stream to the matching ``psk_*``
entry point and raises ``PskError`` on a non-zero status. The shared library is loaded
lazily from this directory on first use and there is no fallback: if ``libpsk.so`` is
missing the call fails with instructions to build it.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from functools import cached_property

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpsk.so")

PSK_F32, PSK_BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "cuda"}
DEV_BAD_BLOCK, DEV_BAD_SEQLEN, DEV_BAD_SELECTED, DEV_BAD_BUDGET, DEV_BAD_APPEND, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10, 0x20

EXPORTS = [
    "psk_kv_append_and_summarize", "psk_page_score_select", "psk_page_score_select_ex", "psk_page_score",
    "psk_page_select", "psk_sparse_paged_decode",
    "psk_sparse_paged_decode_ex", "psk_dense_paged_decode", "psk_sparse_paged_decode_noalloc", "psk_append_workspace_size", "psk_score_select_workspace_size",
    "psk_sparse_decode_workspace_size", "psk_dense_decode_workspace_size", "psk_get_device_status",
    "psk_clear_device_status", "psk_status_string", "psk_version", "psk_selftest_bounded_wait",
    "psk_score_select_launches", "psk_page_select_coverage", "psk_coverage_workspace_size",
    "psk_kv_append_and_summarize_ex", "psk_page_score_select_gaussian", "psk_sparse_paged_decode_tiered",
    "psk_value_tier_fill",
]


class PskError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


class PskLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "v_head_dim", "page_size",
        "num_blocks", "max_pages", "dtype", "latent")]


BUDGET_PER_SEQUENCE, BUDGET_PAGES, BUDGET_FRACTION = 0, 1, 2
DECODE_PER_QUERY_HEAD, DECODE_V_HOST = 0x1, 0x2


class PskSelectParams(ctypes.Structure):
    """Mirrors ``psk_select_params``."""
    _fields_ = [("budgets", ctypes.c_void_p), ("budget_fraction", ctypes.c_double), ("budget_pages", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("sink_pages", ctypes.c_int32), ("window_pages", ctypes.c_int32),
                ("per_query_head", ctypes.c_int32)]


@dataclass(frozen=True)
class Layout:
    """Geometry of one layer's paged cache and decode batch (mirrors ``psk_layout``)."""
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    v_head_dim: int
    page_size: int
    num_blocks: int
    max_pages: int
    dtype: int = PSK_BF16
    latent: int = 0

    def c(self) -> PskLayout:
        return self._c

    @cached_property
    def _c(self) -> PskLayout:  # built once: the layout is frozen and the library only reads it
        return PskLayout(self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim, self.v_head_dim,
                         self.page_size, self.num_blocks, self.max_pages, self.dtype, self.latent)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libpsk.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m page_sparse_kv_gb300.build` "
                               "(or __graft_entry__.build()); there is no non-CUDA fallback")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
        LP = ctypes.POINTER(PskLayout)
        sig = {
            "psk_kv_append_and_summarize": (ctypes.c_int, [LP, P, P, P, P, I, I, P, P, P, P, P, Z, P]),
            "psk_page_score_select": (ctypes.c_int, [LP, P, P, P, P, P, I, F, P, P, P, Z, P]),
            "psk_page_score_select_ex": (ctypes.c_int, [LP, P, P, P, P, ctypes.POINTER(PskSelectParams), I, F, P, P,
                                                        P, Z, P]),
            "psk_sparse_paged_decode": (ctypes.c_int, [LP, P, P, P, P, P, P, I, F, P, P, Z, P]),
            "psk_page_score": (ctypes.c_int, [LP, P, P, P, P, ctypes.POINTER(PskSelectParams), I, F, P, P, Z, P]),
            "psk_page_select": (ctypes.c_int, [LP, P, ctypes.POINTER(PskSelectParams), I, P, P, Z, P]),
            "psk_sparse_paged_decode_ex": (ctypes.c_int, [LP, P, P, P, P, P, P, I, F, ctypes.c_uint32, P, P, Z, P]),
            "psk_dense_paged_decode": (ctypes.c_int, [LP, P, P, P, P, P, F, P, P, Z, P]),
            "psk_sparse_paged_decode_noalloc": (ctypes.c_int, [LP, P, P, P, P, P, P, I, F, P, P]),
            "psk_append_workspace_size": (Z, [LP]),
            "psk_score_select_workspace_size": (Z, [LP, I]),
            "psk_sparse_decode_workspace_size": (Z, [LP, I]),
            "psk_dense_decode_workspace_size": (Z, [LP]),
            "psk_get_device_status": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_uint32), P]),
            "psk_clear_device_status": (ctypes.c_int, [P, P]),
            "psk_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "psk_version": (ctypes.c_int, []),
            "psk_selftest_bounded_wait": (ctypes.c_int, [P, Z, ctypes.c_uint32, P]),
            "psk_score_select_launches": (ctypes.c_int, [LP, I, I]),
            "psk_page_select_coverage": (ctypes.c_int, [LP, P, P, P, P, ctypes.c_double, I, I, I, F, P, P, P, Z, P]),
            "psk_coverage_workspace_size": (Z, [LP, I]),
            "psk_kv_append_and_summarize_ex": (ctypes.c_int, [LP, P, P, P, P, I, I, P, P, P, P, P, P, Z, P]),
            "psk_sparse_paged_decode_tiered": (ctypes.c_int, [LP, P, P, P, P, I, P, P, P, P, I, F, P, P, Z, P]),
            "psk_value_tier_fill": (ctypes.c_int, [LP, P, P, P, I, P, I, P, P, Z, P]),
            "psk_page_score_select_gaussian": (ctypes.c_int, [LP, P, P, P, P, ctypes.POINTER(PskSelectParams), I, F,
                                                              F, P, P, P, Z, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


# ------------------------------------------------------------------------------ helpers
def _ptr(t):
    """Device-addressable pointer of a contiguous tensor: a CUDA tensor, or a pinned host tensor
    (under unified addressing the GPU reads and writes it by its host pointer, e.g. the value
    cache of the host-memory value tier)."""
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("expected a CUDA tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


_current_raw_stream = None


def _stream(stream):
    """cudaStream_t of `stream`, or of torch's current stream on the current device. The
    current one comes from torch's raw-stream query when it has one (about 10x cheaper per
    call than building a torch.cuda.Stream object), else from torch.cuda.current_stream()."""
    global _current_raw_stream
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _current_raw_stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and dev is not None:
            _current_raw_stream = lambda: raw(dev())
        else:
            _current_raw_stream = lambda: torch.cuda.current_stream().cuda_stream
    return ctypes.c_void_p(_current_raw_stream())


def _check(fn: str, code: int):
    if code != 0:
        msg = lib().psk_status_string(code).decode()
        raise PskError(fn, code, msg)


def storage_dtype(layout: Layout):
    import torch
    return torch.float32 if layout.dtype == PSK_F32 else torch.bfloat16


# ------------------------------------------------------------------------------ sizes
def append_workspace_size(layout: Layout) -> int:
    return int(lib().psk_append_workspace_size(ctypes.byref(layout.c())))


def score_select_workspace_size(layout: Layout, b_max: int) -> int:
    return int(lib().psk_score_select_workspace_size(ctypes.byref(layout.c()), int(b_max)))


def sparse_decode_workspace_size(layout: Layout, b_max: int) -> int:
    return int(lib().psk_sparse_decode_workspace_size(ctypes.byref(layout.c()), int(b_max)))


def dense_decode_workspace_size(layout: Layout) -> int:
    return int(lib().psk_dense_decode_workspace_size(ctypes.byref(layout.c())))


def score_select_launches(layout: Layout, b_max: int, per_query_head: bool = False) -> int:
    """Kernel launches of one page_score_select(_ex) call (1: selection fused into the score
    kernel, 2: a separate selection launch, 3: latent form); 0 if unsupported."""
    return int(lib().psk_score_select_launches(ctypes.byref(layout.c()), int(b_max), 1 if per_query_head else 0))


def coverage_workspace_size(layout: Layout, b_max: int) -> int:
    return int(lib().psk_coverage_workspace_size(ctypes.byref(layout.c()), int(b_max)))


def workspace_size(layout: Layout, b_max: int, coverage: bool = False) -> int:
    """Bytes of one workspace that serves every call of this layout and budget bound (and the
    coverage selection when ``coverage``)."""
    sizes = [append_workspace_size(layout), score_select_workspace_size(layout, b_max),
             sparse_decode_workspace_size(layout, b_max), dense_decode_workspace_size(layout)]
    if coverage:
        sizes.append(coverage_workspace_size(layout, b_max))
    if min(sizes) == 0:
        raise PskError("workspace_size", 2, "layout not supported")
    return max(sizes)


def make_workspace(layout: Layout, b_max: int, device=None, coverage: bool = False):
    """A zero-filled workspace tensor (uint8) sized for every call of this layout."""
    import torch
    return torch.zeros(workspace_size(layout, b_max, coverage), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------------------ calls
def kv_append_and_summarize(layout: Layout, k_new, v_new, start_pos, cu_new, max_new: int, k_cache, v_cache,
                            summaries, block_table, workspace, stream=None):
    total_new = int(k_new.shape[0]) if k_new is not None else 0
    _check("psk_kv_append_and_summarize", lib().psk_kv_append_and_summarize(
        ctypes.byref(layout.c()), _ptr(k_new), _ptr(v_new), _ptr(start_pos), _ptr(cu_new), total_new,
        int(max_new), _ptr(k_cache), _ptr(v_cache), _ptr(summaries), _ptr(block_table), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def kv_append_and_summarize_ex(layout: Layout, k_new, v_new, start_pos, cu_new, max_new: int, k_cache, v_cache,
                               summaries, stats, block_table, workspace, stream=None):
    """kv_append_and_summarize that also (or only) keeps the fp32 per-page key mean / std store
    ``stats`` [num_blocks, num_kv_heads, 2, head_dim]; either store may be None, not both."""
    total_new = int(k_new.shape[0]) if k_new is not None else 0
    _check("psk_kv_append_and_summarize_ex", lib().psk_kv_append_and_summarize_ex(
        ctypes.byref(layout.c()), _ptr(k_new), _ptr(v_new), _ptr(start_pos), _ptr(cu_new), total_new,
        int(max_new), _ptr(k_cache), _ptr(v_cache), _ptr(summaries), _ptr(stats), _ptr(block_table),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def page_score_select_gaussian(layout: Layout, q, stats, block_table, seq_lens, b_max: int, scale: float, z: float,
                               selected, workspace, *, budgets=None, budget_pages: int | None = None,
                               budget_fraction: float | None = None, sink_pages: int = 1, window_pages: int = 1,
                               scores_out=None, stream=None):
    """Top-b pages by the Gaussian estimated maximum from the mean / std store (see psk.h)."""
    prm = select_params(budgets=budgets, budget_pages=budget_pages, budget_fraction=budget_fraction,
                        sink_pages=sink_pages, window_pages=window_pages)
    _check("psk_page_score_select_gaussian", lib().psk_page_score_select_gaussian(
        ctypes.byref(layout.c()), _ptr(q), _ptr(stats), _ptr(block_table), _ptr(seq_lens), ctypes.byref(prm),
        int(b_max), float(scale), float(z), _ptr(selected), _ptr(scores_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def page_score_select(layout: Layout, q, summaries, block_table, seq_lens, budgets, b_max: int, scale: float,
                      selected, workspace, scores_out=None, stream=None):
    _check("psk_page_score_select", lib().psk_page_score_select(
        ctypes.byref(layout.c()), _ptr(q), _ptr(summaries), _ptr(block_table), _ptr(seq_lens), _ptr(budgets),
        int(b_max), float(scale), _ptr(selected), _ptr(scores_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def select_params(*, budgets=None, budget_pages: int | None = None, budget_fraction: float | None = None,
                  sink_pages: int = 1, window_pages: int = 1, per_query_head: bool = False) -> PskSelectParams:
    """A ``psk_select_params`` with exactly one budget mode (see ``page_score_select_ex``)."""
    modes = [budgets is not None, budget_pages is not None, budget_fraction is not None]
    if sum(modes) != 1:
        raise ValueError("give exactly one of budgets, budget_pages, budget_fraction")
    prm = PskSelectParams()
    prm.budgets = _ptr(budgets) if budgets is not None else None
    prm.budget_fraction = float(budget_fraction or 0.0)
    prm.budget_pages = int(budget_pages or 0)
    prm.mode = BUDGET_PER_SEQUENCE if modes[0] else (BUDGET_PAGES if modes[1] else BUDGET_FRACTION)
    prm.sink_pages, prm.window_pages = int(sink_pages), int(window_pages)
    prm.per_query_head = 1 if per_query_head else 0
    return prm


def page_score(layout: Layout, q, summaries, block_table, seq_lens, params: PskSelectParams, b_max: int,
               scale: float, workspace, scores_out=None, stream=None):
    """Stage 2 alone: selection keys into ``workspace`` (and scores into ``scores_out``)."""
    _check("psk_page_score", lib().psk_page_score(
        ctypes.byref(layout.c()), _ptr(q), _ptr(summaries), _ptr(block_table), _ptr(seq_lens), ctypes.byref(params),
        int(b_max), float(scale), _ptr(scores_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def page_select(layout: Layout, seq_lens, params: PskSelectParams, b_max: int, selected, workspace, stream=None):
    """Stage 3 alone: the selected rows from the keys ``page_score`` left in ``workspace``."""
    _check("psk_page_select", lib().psk_page_select(
        ctypes.byref(layout.c()), _ptr(seq_lens), ctypes.byref(params), int(b_max), _ptr(selected), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def page_score_select_ex(layout: Layout, q, summaries, block_table, seq_lens, b_max: int, scale: float, selected,
                         workspace, *, budgets=None, budget_pages: int | None = None,
                         budget_fraction: float | None = None, sink_pages: int = 1, window_pages: int = 1,
                         per_query_head: bool = False, scores_out=None, stream=None):
    """Score + select with the first ``sink_pages`` and last ``window_pages`` pages always kept
    and exactly one budget mode: ``budgets`` (device int32 per sequence), ``budget_pages`` (a
    fixed page count) or ``budget_fraction`` (a fraction of each sequence's pages). With
    ``per_query_head`` the rows are per (sequence, query head): ``selected`` is
    [batch, num_q_heads, b_max]."""
    prm = select_params(budgets=budgets, budget_pages=budget_pages, budget_fraction=budget_fraction,
                        sink_pages=sink_pages, window_pages=window_pages, per_query_head=per_query_head)
    _check("psk_page_score_select_ex", lib().psk_page_score_select_ex(
        ctypes.byref(layout.c()), _ptr(q), _ptr(summaries), _ptr(block_table), _ptr(seq_lens), ctypes.byref(prm),
        int(b_max), float(scale), _ptr(selected), _ptr(scores_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def page_select_coverage(layout: Layout, q, k_cache, block_table, seq_lens, coverage: float, b_max: int,
                         scale: float, selected, workspace, sink_pages: int = 1, window_pages: int = 1,
                         masses_out=None, stream=None):
    """Adaptive per-head coverage: the always-kept pages plus the fewest highest-mass pages whose
    exact softmax mass reaches ``coverage`` of the unit's total (see psk.h); rows into
    ``selected`` [batch, num_kv_heads, b_max], masses into ``masses_out`` when given."""
    _check("psk_page_select_coverage", lib().psk_page_select_coverage(
        ctypes.byref(layout.c()), _ptr(q), _ptr(k_cache), _ptr(block_table), _ptr(seq_lens), float(coverage),
        int(sink_pages), int(window_pages), int(b_max), float(scale), _ptr(selected), _ptr(masses_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def sparse_paged_decode(layout: Layout, q, k_cache, v_cache, block_table, seq_lens, selected, b_max: int,
                        scale: float, out, workspace, stream=None):
    _check("psk_sparse_paged_decode", lib().psk_sparse_paged_decode(
        ctypes.byref(layout.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(selected), int(b_max), float(scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def sparse_paged_decode_ex(layout: Layout, q, k_cache, v_cache, block_table, seq_lens, selected, b_max: int,
                           scale: float, out, workspace, per_query_head: bool = False, v_host: bool = False,
                           stream=None):
    """sparse_paged_decode over rows per (sequence, query head) when ``per_query_head``; with
    ``v_host`` the value cache is a pinned host tensor read over NVLink-C2C."""
    flags = (DECODE_PER_QUERY_HEAD if per_query_head else 0) | (DECODE_V_HOST if v_host else 0)
    _check("psk_sparse_paged_decode_ex", lib().psk_sparse_paged_decode_ex(
        ctypes.byref(layout.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(selected), int(b_max), float(scale), flags, _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def sparse_paged_decode_tiered(layout: Layout, q, k_cache, v_cache_host, v_hot, v_slot, block_table, seq_lens,
                               selected, b_max: int, scale: float, out, workspace, stream=None):
    """Sparse decode with V in pinned host memory and the pages that have a slot in ``v_slot``
    read from the resident HBM copies ``v_hot`` [n_slots, page_size, head_dim] (see psk.h)."""
    _check("psk_sparse_paged_decode_tiered", lib().psk_sparse_paged_decode_tiered(
        ctypes.byref(layout.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache_host), _ptr(v_hot), int(v_hot.shape[0]),
        _ptr(v_slot), _ptr(block_table), _ptr(seq_lens), _ptr(selected), int(b_max), float(scale), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def value_tier_fill(layout: Layout, v_cache_host, block_table, entries, v_hot, v_slot, workspace, stream=None):
    """Fill / evict hot-buffer slots: entries int32 [n, 4] of (sequence, KV head, page, slot), slot < 0
    evicts (see psk.h)."""
    n = 0 if entries is None else int(entries.shape[0])
    _check("psk_value_tier_fill", lib().psk_value_tier_fill(
        ctypes.byref(layout.c()), _ptr(v_cache_host), _ptr(block_table), _ptr(entries) if n else None, n,
        _ptr(v_hot), int(v_hot.shape[0]), _ptr(v_slot), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def dense_paged_decode(layout: Layout, q, k_cache, v_cache, block_table, seq_lens, scale: float, out, workspace,
                       stream=None):
    _check("psk_dense_paged_decode", lib().psk_dense_paged_decode(
        ctypes.byref(layout.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        float(scale), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def sparse_paged_decode_noalloc(layout: Layout, q, k_cache, v_cache, block_table, seq_lens, selected, b_max: int,
                                scale: float, out, stream=None):
    """sparse_paged_decode without a workspace, for callers that cannot allocate device memory:
    the library's fixed 32 MiB per-device scratch holds the split partials (see psk.h)."""
    _check("psk_sparse_paged_decode_noalloc", lib().psk_sparse_paged_decode_noalloc(
        ctypes.byref(layout.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(selected), int(b_max), float(scale), _ptr(out), _stream(stream)))


def get_device_status(workspace, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check("psk_get_device_status", lib().psk_get_device_status(_ptr(workspace), ctypes.byref(v), _stream(stream)))
    return int(v.value)


def clear_device_status(workspace, stream=None):
    _check("psk_clear_device_status", lib().psk_clear_device_status(_ptr(workspace), _stream(stream)))


def selftest_bounded_wait(workspace, spin_limit: int, stream=None):
    """Runs the kernels' bounded wait on a phase that never completes (see psk.h): afterwards
    the workspace status word holds DEV_TIMEOUT."""
    _check("psk_selftest_bounded_wait", lib().psk_selftest_bounded_wait(
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(spin_limit), _stream(stream)))


def version() -> int:
    return int(lib().psk_version())
