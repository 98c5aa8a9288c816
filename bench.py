#!/usr/bin/env python3
"""Decode-step benchmark of page-selective sparse paged attention on one GB300 (per rank).

One step = the whole hot path over one batch: append one decode token per sequence with its
page-summary refresh, score + select pages, sparse split-K decode (4 kernel launches; 5 on the
latent config). The step's launches are captured once into a CUDA graph and the reported value
is the mean over K graph replays (CUDA events on the launching stream); the same window also
times the eager launches (with a per-call split) and the dense step (append + full-KV decode)
both ways, so the speedup compares like with like.

Default workload: batched ragged decode, B=64, H_q=32, H_kv=8, D=128, page 16, contexts
U[8192, 65536], bf16, budget max(4, ceil(5% of pages)), 16 hot pages per KV head.
Inputs stay larger than L2 every step (summaries ~0.6 GB, selected K/V ~0.5 GB in a 9.7 GB
pool), so no L2 flush is needed.

    python bench.py [--steps K] [--warmup W] [--impl psk|reference] [--workload 1..5]
    torchrun --nproc-per-node N bench.py --gpus N      # N independent replicas (weak scaling)
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import math
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode µs/step/layer; achieved HBM GB/s vs GB300 peak; speedup vs dense"
UNIT = "us/step/layer"


def peaks():
    """HBM GB/s and bf16 TFLOP/s (burst, sustained) measured on this GPU model, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "kind": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "kind": "fallback"}


# DRAM bytes (read + write) per launch of the dominant call, from one ncu capture of that call
# (dram__bytes_read.sum + dram__bytes_write.sum, summed over its kernels), keyed by workload and
# call, with a digest of the sources the kernels are built from: a digest that no longer matches
# means the kernels changed since the capture, and the traffic is reported as null.
TRAFFIC = {
    # One-pass capture on the first 16 sequences (profiles/page_score_mma_kernel_batched_ragged_b16.md):
    #   python bench.py --batch 16 --steps 3 --warmup 3 --no-cpu-baseline, then
    #   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum --clock-control none
    #       -k regex:"page_score|page_select|decode_split" -s 0 -c 3 python bench.py --batch 16 --steps 3 ...
    # 158,038,272 + 2,779,904 B for 38,540 pages; scaled by pages to the 140,808 of the full workload.
    ("batched-ragged-b64-8k..64k-5pct", "page_score_mma_kernel"):
        {"bytes": 587_558_011, "digest": "fee1dcb211b0b4f0", "scaled_from": "first 16 sequences, by pages"},
    # 129,188,864 + 2,953,728 B for 15,472 selected (page, head) pairs (ncu -k regex:decode_split
    # -s 0 -c 1, the same command otherwise); 56,536 in the full workload
    ("batched-ragged-b64-8k..64k-5pct", "decode_split_kernel"):
        {"bytes": 482_860_237, "digest": "b3d841046fbd5db0", "scaled_from": "first 16 sequences, by selected pages"},
}
KERNEL_SOURCES = {
    "page_score_kernel": ("score_select.cu", "psk_common.cuh", "psk_internal.h"),
    "page_score_mma_kernel": ("score_select.cu", "psk_common.cuh", "psk_internal.h"),
    "page_select_kernel": ("select.cu", "select_common.cuh", "psk_common.cuh", "psk_internal.h"),
    "decode_split_kernel": ("decode.cu", "psk_common.cuh", "psk_internal.h"),
    "mla_qsplit_kernel+mla_score_kernel": ("mla.cu", "psk_common.cuh", "psk_internal.h"),
    "mla_decode_kernel": ("mla.cu", "psk_common.cuh", "psk_internal.h"),
}


def kernel_digest(call: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[call]:
        with open(os.path.join(ROOT, "page_sparse_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(workload: str, call: str):
    rec = TRAFFIC.get((workload, call))
    if rec is None or rec["digest"] != kernel_digest(call):
        return None, None
    return rec["bytes"], rec.get("scaled_from")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ------------------------------------------------------------------------------------------
def max_over_ranks(values, device):
    """Element-wise max of per-rank timings over the process group (the slowest replica sets
    the step time). NaN (a mode a rank could not run) stays NaN."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    nan = torch.isnan(t).to(torch.float64)
    dist.all_reduce(nan, op=dist.ReduceOp.MAX)
    t = torch.nan_to_num(t, nan=0.0)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    t[nan > 0] = float("nan")
    return t.tolist()


def _oracle_worker(workload: int, batch: int, units, n_steps: int, seconds: float, barrier, results):
    """One host core's share of the oracle baseline: the oracle's sparse decode step (score every
    page, select, attend) over this worker's (sequence, KV head) units, repeated for ``seconds``
    per timed step. A unit is the oracle's functions applied to that KV head's slice of the
    sequence (its query heads, keys, values and summaries). Page summaries and inputs are
    prepared before the timed steps (they are cache state the append step maintains). Puts
    [(seconds, unit pages), ...] per step on ``results``."""
    import oracle as O
    import workloads as W
    w = W.config(workload)
    if batch and batch < w.B:
        w = W.prefix(w, batch)
    scale = 1.0 / math.sqrt(w.D)
    G = w.H_q // w.H_kv
    prep = []
    for i in sorted({u[0] for u in units}):
        L = int(w.seq_lens[i])
        keys, vals, q = w.keys(i), w.values(i), w.query(i)
        for h in sorted(u[1] for u in units if u[0] == i):
            k_h = np.ascontiguousarray(keys[:, h:h + 1])
            v_h = np.ascontiguousarray(vals[:, h:h + 1])
            kmin, kmax = O.page_summaries(k_h, L, w.page_size, w.dtype)
            prep.append((i, L, k_h, v_h, kmin, kmax, np.ascontiguousarray(q[h * G:(h + 1) * G])))
        del keys, vals
    out = []
    for _ in range(n_steps):
        barrier.wait(timeout=1800)
        t0 = time.perf_counter()
        pages, k = 0, 0
        while True:
            i, L, k_h, v_h, kmin, kmax, q_h = prep[k % len(prep)]
            s = O.quest_scores(q_h, kmin, kmax, w.dtype, scale)
            sel = [O.select_pages(s[0], int(w.budgets[i]))]
            O.attend_pages(q_h, k_h, v_h, L, w.page_size, sel, w.dtype, scale)
            pages += -(-L // w.page_size)
            k += 1
            if time.perf_counter() - t0 >= seconds:
                break
        out.append((time.perf_counter() - t0, pages))
    results.put(out)


def oracle_parallel(workload: int, batch: int, n_steps: int, seconds: float):
    """Times the fp64 oracle's sparse step on every host core this process may use: one spawned
    process per core, each holding a contiguous share of the batch's (sequence, KV head) units;
    every step is a window of about ``seconds`` in which all workers run at once (a barrier
    starts it). A step's time is the batch's unit pages divided by the rate of the window (all
    workers' unit pages over the slowest worker's time). Returns (per-step seconds for the
    whole batch, cores, sequence-steps)."""
    import multiprocessing as mp
    import workloads as W
    w = W.config(workload)
    if batch and batch < w.B:
        w = W.prefix(w, batch)
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    units = [(i, h) for i in range(w.B) for h in range(w.H_kv)]
    n = max(1, min(cores, len(units)))
    shares = [units[j * len(units) // n:(j + 1) * len(units) // n] for j in range(n)]
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(workload, batch, shares[j], n_steps, seconds, barrier, results))
             for j in range(n)]
    for pr in procs:
        pr.start()
    outs = [results.get(timeout=3600) for _ in procs]
    for pr in procs:
        pr.join(timeout=60)
    total_pages = int(((w.seq_lens + w.page_size - 1) // w.page_size).sum()) * w.H_kv
    per_step = []
    seq_steps = 0
    for s in range(n_steps):
        t = max(o[s][0] for o in outs)
        pg = sum(o[s][1] for o in outs)
        per_step.append(total_pages / (pg / t))
        seq_steps += round(pg / (total_pages / w.B))
    return per_step, n, seq_steps


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads as W
    w = W.config(args.workload)
    per_step_s = max(0.3, args.ref_seconds / max(1, args.steps + args.warmup))  # the whole run: ref_seconds of windows
    times, cores, seqs = oracle_parallel(args.workload, 0, args.warmup + args.steps, per_step_s)
    times = times[args.warmup:]
    us = statistics.mean(times) * 1e6
    sample = (f"about {seqs} sequence-steps (in pages) of the fp64 oracle's sparse step (score all pages, select, "
              f"attend), {cores} processes on {cores} host cores, {per_step_s:.2f} s windows, scaled to the "
              f"{w.B}-sequence batch by pages")
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "D": w.D,
                       "page_size": w.page_size, "budget": "max(4, ceil(5% of pages))"},
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
def run_psk(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    import __graft_entry__
    __graft_entry__.build()
    import page_sparse_kv_gb300 as psk
    import workloads as W
    from workloads.device import budgets as dev_budgets, to_torch, upload

    w = W.config(args.workload)
    if args.batch and args.batch < w.B:
        w = W.prefix(w, args.batch)
    t_setup = time.time()
    cache = upload(w)
    L = cache.layout
    B, Hq, Hkv, D = w.B, w.H_q, w.H_kv, w.D
    es = w.elem_bytes
    dev = cache.device
    stream = torch.cuda.current_stream()

    # the decode token of every sequence: its last token (re-appended in place each step, so the
    # cache state is identical before and after a step)
    lens = w.seq_lens.astype(np.int64)
    k_last = np.stack([w.keys(i, int(lens[i]) - 1, int(lens[i]))[0] for i in range(B)])
    v_last = None if w.latent else np.stack([w.values(i, int(lens[i]) - 1, int(lens[i]))[0] for i in range(B)])
    q_host = w.queries()
    k_new = to_torch(k_last, w.dtype).to(dev)
    v_new = None if w.latent else to_torch(v_last, w.dtype).to(dev)
    q = to_torch(q_host, w.dtype).to(dev)
    start = torch.from_numpy((lens - 1).astype(np.int32)).to(dev)
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev)
    bud = dev_budgets(w)
    sel = torch.empty(B, Hkv, w.b_max, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, w.D_v, dtype=cache.dtype, device=dev)
    out_dense = torch.empty_like(out)
    ws = cache.ws
    setup_s = time.time() - t_setup

    # --v-host: the value tier in pinned host memory, read (and appended to) over NVLink-C2C;
    # --v-hot F: plus a resident HBM hot buffer holding the fraction F of each row's selected pages
    # (filled after the warm-up from that step's selection, which the timed steps repeat)
    v_store = cache.v_cache.cpu().pin_memory() if args.v_host else cache.v_cache
    hot = None
    if args.v_host and (w.latent or w.dtype != "bf16" or D != 128):
        raise SystemExit("--v-host is built for GQA bf16 caches with head_dim 128")
    selector = args.selector
    if selector != "bound" and (w.latent or args.v_host):
        raise SystemExit("--selector other than bound is built for GQA caches with V in HBM")
    if selector == "per-query-head":  # one selected row per query head
        sel = torch.empty(B, Hq, w.b_max, dtype=torch.int32, device=dev)
    if selector == "coverage":  # the K-only mass pass needs the coverage workspace
        ws = psk.make_workspace(L, w.b_max, dev, coverage=True)
    stats = None
    if selector == "gaussian":
        # the fp32 key mean / std store, built (untimed) by re-appending every sequence's keys and
        # values from the cache itself, a few sequences at a time
        stats = torch.zeros(w.num_blocks, Hkv, 2, D, dtype=torch.float32, device=dev)
        bt_dev = cache.block_table
        for i0 in range(0, B, 4):
            idx = list(range(i0, min(B, i0 + 4)))
            ks, vs, cu_l = [], [], [0]
            for i in idx:
                n = int(lens[i])
                P_i = (n + w.page_size - 1) // w.page_size
                blocks = bt_dev[i, :P_i].long()
                ks.append(cache.k_cache[blocks].reshape(-1, Hkv, D)[:n])
                vs.append(cache.v_cache[blocks].reshape(-1, Hkv, w.D_v)[:n])
                cu_l.append(cu_l[-1] + n)
            cu_i = torch.tensor(cu_l, dtype=torch.int32, device=dev)
            st_i = torch.zeros(len(idx), dtype=torch.int32, device=dev)
            Li = psk.Layout(len(idx), Hq, Hkv, D, w.D_v, w.page_size, w.num_blocks, w.max_pages, L.dtype, L.latent)
            psk.kv_append_and_summarize_ex(Li, torch.cat(ks), torch.cat(vs), st_i, cu_i, max(cu_l[j + 1] - cu_l[j]
                                           for j in range(len(idx))), cache.k_cache, cache.v_cache, None, stats,
                                           bt_dev[i0:i0 + len(idx)].contiguous(), ws)
            del ks, vs
        torch.cuda.synchronize()

    def append():
        if stats is not None:  # both stores kept in step
            psk.kv_append_and_summarize_ex(L, k_new, v_new, start, cu, 1, cache.k_cache, v_store, cache.summaries,
                                           stats, cache.block_table, ws)
        else:
            psk.kv_append_and_summarize(L, k_new, v_new, start, cu, 1, cache.k_cache, v_store, cache.summaries,
                                        cache.block_table, ws)

    def score():
        if selector == "per-query-head":
            psk.page_score_select_ex(L, q, cache.summaries, cache.block_table, cache.seq_lens, w.b_max, cache.scale,
                                     sel, ws, budgets=bud, per_query_head=True)
        elif selector == "coverage":
            psk.page_select_coverage(L, q, cache.k_cache, cache.block_table, cache.seq_lens, args.coverage, w.b_max,
                                     cache.scale, sel, ws)
        elif selector == "gaussian":
            psk.page_score_select_gaussian(L, q, stats, cache.block_table, cache.seq_lens, w.b_max, cache.scale,
                                           args.gauss_z, sel, ws, budgets=bud)
        else:
            psk.page_score_select(L, q, cache.summaries, cache.block_table, cache.seq_lens, bud, w.b_max,
                                  cache.scale, sel, ws)

    # kernels one score + select call launches: 2 (score, selection), 3 for the latent form and
    # for coverage (mass pass, keys and count, selection)
    ss_launches = 3 if selector == "coverage" else psk.score_select_launches(L, w.b_max,
                                                                             selector == "per-query-head")

    # the same two stages as separate calls, so each kernel gets its own events in the eager loop
    # (coverage and the Gaussian score are one call each: timed as the score, selection included)
    sel_prm = psk.select_params(budgets=bud, per_query_head=selector == "per-query-head")

    def score_only():
        if selector in ("coverage", "gaussian"):
            score()
        else:
            psk.page_score(L, q, cache.summaries, cache.block_table, cache.seq_lens, sel_prm, w.b_max, cache.scale,
                           ws)

    def select_only():
        if selector not in ("coverage", "gaussian"):
            psk.page_select(L, cache.seq_lens, sel_prm, w.b_max, sel, ws)

    def decode(dst=None):  # dst: the output buffer (default: `out` in device memory)
        o = out if dst is None else dst
        if args.v_host and hot is not None:
            psk.sparse_paged_decode_tiered(L, q, cache.k_cache, v_store, hot[0], hot[1], cache.block_table,
                                           cache.seq_lens, sel, w.b_max, cache.scale, o, ws)
        elif args.v_host:
            psk.sparse_paged_decode_ex(L, q, cache.k_cache, v_store, cache.block_table, cache.seq_lens, sel, w.b_max,
                                       cache.scale, o, ws, v_host=True)
        elif selector == "per-query-head":
            psk.sparse_paged_decode_ex(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, sel,
                                       w.b_max, cache.scale, o, ws, per_query_head=True)
        else:
            psk.sparse_paged_decode(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, sel,
                                    w.b_max, cache.scale, o, ws)

    def dense():
        psk.dense_paged_decode(L, q, cache.k_cache, cache.v_cache, cache.block_table, cache.seq_lens, cache.scale,
                               out_dense, ws)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    launches_per_step = 2 + ss_launches  # append, score (+ select, + q split), decode
    for _ in range(args.warmup):
        append(); score(); decode()
        append(); dense()
    torch.cuda.synchronize()
    assert psk.get_device_status(ws) == 0, "device status set during warm-up"
    hot_pages = 0
    if args.v_host and args.v_hot > 0:
        sel_np = sel.cpu().numpy()
        ents = []
        for i in range(B):
            for h in range(Hkv):
                row = [int(x) for x in sel_np[i, h] if x >= 0]
                ents += [(i, h, p) for p in row[:int(round(len(row) * args.v_hot))]]
        hot_pages = len(ents)
        v_hot = torch.empty(max(1, hot_pages), w.page_size, D, dtype=cache.dtype, device=dev)
        v_slot = torch.full((B, Hkv, w.max_pages), -1, dtype=torch.int32, device=dev)
        if ents:
            e_t = torch.tensor([(i, h, p, k) for k, (i, h, p) in enumerate(ents)], dtype=torch.int32, device=dev)
            psk.value_tier_fill(L, v_store, cache.block_table, e_t, v_hot, v_slot, ws)
        hot = (v_hot, v_slot)
        append(); score(); decode()
        torch.cuda.synchronize()
        assert psk.get_device_status(ws) == 0, "device status set by the hot-buffer fill"

    # ---- the same steps captured once into CUDA graphs (replayed inside the timed window) ------
    # The one-token append touches only the tail page, whose summary the score call does not
    # read (the tail is kept whatever its score): the graphed step runs the append on a side
    # stream beside score + select, and the decode waits for both (page_sparse_kv_gb300.step,
    # the same step tests/test_gpu_step_graph.py checks against the oracle).
    from page_sparse_kv_gb300.step import DecodeStep, capture as graph_of
    # coverage reads every key row (the tail page's too) and the Gaussian score reads the tail
    # page's statistics: there the append runs before the selection on the main stream
    if selector in ("coverage", "gaussian"):
        sparse_step = DecodeStep(lambda: None, lambda: (append(), score()), decode)
    else:
        sparse_step = DecodeStep(append, score, decode)

    def step_overlapped(pre_main=None, pre_side=None, post=None, dec_out=None):
        if dec_out is None:
            sparse_step.launch(pre_main, pre_side, post)
        else:
            DecodeStep(sparse_step.append, sparse_step.score_select, lambda: decode(dec_out)).launch(
                pre_main, pre_side, post)

    try:
        g_sparse = graph_of(step_overlapped)
        g_dense = graph_of(lambda: (append(), dense()))
        for _ in range(3):
            g_sparse.replay()
            g_dense.replay()
        torch.cuda.synchronize()
    except Exception as exc:  # capture not possible here: report eager numbers only
        print(f"graph capture failed: {exc}", file=sys.stderr)
        g_sparse = g_dense = None

    # ---- timed region: eager steps with per-kernel events, dense steps, graph replays ----------
    # A step whose working set (summaries + selected K/V + q/out; every page for the dense step)
    # is under four times L2 would run from L2 when repeated: then L2 is flushed (a buffer of
    # twice its size is written) before every timed step, outside that step's events.
    try:
        l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        l2 = 126 << 20
    lens64 = w.seq_lens.astype(np.int64)
    P_est = (lens64 + w.page_size - 1) // w.page_size
    kv_row_est = D if w.latent else D + w.D_v
    ws_sparse = int(P_est.sum()) * Hkv * 2 * D * es + int(np.minimum(w.budgets, P_est).sum()) * Hkv * w.page_size * kv_row_est * es
    ws_dense = int(lens64.sum()) * Hkv * kv_row_est * es
    flush = ws_sparse < 4 * l2 or ws_dense < 4 * l2
    fbuf = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev) if flush else None

    def flush_l2():
        if fbuf is not None:
            fbuf.fill_(0)

    K = args.steps
    Kd = max(3, K // 4)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    evd = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kd)]
    evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    evgd = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kd)]
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    barrier()
    clk = Clocks(local)  # samples through the timed windows below, the end-to-end one included
    clk.__enter__()
    marks[0].record(stream)
    for k in range(K):
        flush_l2()
        e = ev[k]
        e[0].record(stream)
        append()
        e[1].record(stream)
        score_only()
        e[2].record(stream)
        select_only()
        e[3].record(stream)
        decode()
        e[4].record(stream)
    marks[1].record(stream)
    for k in range(Kd):
        flush_l2()
        evd[k][0].record(stream)
        append(); dense()
        evd[k][1].record(stream)
    marks[2].record(stream)
    if g_sparse is not None:
        marks[3].record(stream)
        for k in range(K):
            flush_l2()
            evg[k][0].record(stream)
            g_sparse.replay()
            evg[k][1].record(stream)
        marks[4].record(stream)
        for k in range(Kd):
            flush_l2()
            evgd[k][0].record(stream)
            g_dense.replay()
            evgd[k][1].record(stream)
        marks[5].record(stream)
    torch.cuda.synchronize()
    barrier()

    def per_step(pairs):
        return statistics.mean(x[0].elapsed_time(x[-1]) for x in pairs)

    if flush:  # per-step events: the flushes between them are not timed
        sparse_ms, dense_ms = per_step(ev), per_step(evd)
        graph_sparse_ms = per_step(evg) if g_sparse is not None else float("nan")
        graph_dense_ms = per_step(evgd) if g_sparse is not None else float("nan")
    else:  # back-to-back steps: the window over K steps
        sparse_ms = marks[0].elapsed_time(marks[1]) / K
        dense_ms = marks[1].elapsed_time(marks[2]) / Kd
        if g_sparse is not None:
            graph_sparse_ms = marks[3].elapsed_time(marks[4]) / K
            graph_dense_ms = marks[4].elapsed_time(marks[5]) / Kd
        else:
            graph_sparse_ms = graph_dense_ms = float("nan")
    t_app = statistics.mean(ev[k][0].elapsed_time(ev[k][1]) for k in range(K))
    t_score = statistics.mean(ev[k][1].elapsed_time(ev[k][2]) for k in range(K))
    t_select = statistics.mean(ev[k][2].elapsed_time(ev[k][3]) for k in range(K))
    t_dec = statistics.mean(ev[k][3].elapsed_time(ev[k][4]) for k in range(K))
    if dist is not None:
        sparse_ms, dense_ms, graph_sparse_ms, graph_dense_ms = max_over_ranks(
            [sparse_ms, dense_ms, graph_sparse_ms, graph_dense_ms], dev)

    # ---- end to end: host buffers through the C ABI. The step's inputs are copied from pinned
    # host memory (H2D); the decode writes its output straight into the pinned host buffer (the
    # GPU addresses it under unified addressing, the bytes cross NVLink-C2C inside the step)
    qh = to_torch(q_host, w.dtype).pin_memory()
    kh = to_torch(k_last, w.dtype).pin_memory()
    vh = None if w.latent else to_torch(v_last, w.dtype).pin_memory()
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    Ke = max(3, K // 4)
    for _ in range(2):
        q.copy_(qh, non_blocking=True); k_new.copy_(kh, non_blocking=True)
        if vh is not None:
            v_new.copy_(vh, non_blocking=True)
        append(); score(); decode(oh)
    barrier()
    exs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    for k in range(Ke):
        flush_l2()
        exs[k][0].record(stream)
        q.copy_(qh, non_blocking=True); k_new.copy_(kh, non_blocking=True)
        if vh is not None:
            v_new.copy_(vh, non_blocking=True)
        append(); score(); decode(oh)
        exs[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_eager_ms = per_step(exs)

    def e2e_step():
        def copy_kv():
            k_new.copy_(kh, non_blocking=True)
            if vh is not None:
                v_new.copy_(vh, non_blocking=True)
        if selector in ("coverage", "gaussian"):  # the append runs on the main stream: copy there
            step_overlapped(pre_main=lambda: (q.copy_(qh, non_blocking=True), copy_kv()), dec_out=oh)
        else:
            step_overlapped(pre_main=lambda: q.copy_(qh, non_blocking=True), pre_side=copy_kv, dec_out=oh)

    e2e_ms = e2e_eager_ms
    if g_sparse is not None:  # the same step with its copies, replayed as one CUDA graph
        try:
            g_e2e = graph_of(e2e_step)
            for _ in range(3):
                g_e2e.replay()
            barrier()
            eys = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
            for k in range(Ke):
                flush_l2()
                eys[k][0].record(stream)
                g_e2e.replay()
                eys[k][1].record(stream)
            torch.cuda.synchronize()
            e2e_ms = per_step(eys)
        except Exception as exc:
            print(f"graph capture of the end-to-end step failed: {exc}", file=sys.stderr)
    clk.__exit__(None, None, None)
    if dist is not None:
        e2e_ms, e2e_eager_ms = max_over_ranks([e2e_ms, e2e_eager_ms], dev)
    h2d = (qh.numel() + kh.numel() + (0 if vh is None else vh.numel())) * es
    d2h = oh.numel() * es
    assert psk.get_device_status(ws) == 0, "device status set during the timed region"

    # ---- algorithmic bytes --------------------------------------------------------------------
    P = (lens + w.page_size - 1) // w.page_size
    summ_bytes = int(P.sum()) * Hkv * 2 * D * es
    q_bytes = B * Hq * D * es
    out_bytes = B * Hq * w.D_v * es
    kv_row = D if w.latent else D + w.D_v  # a latent row carries the value in its first D_v dims
    sel_np = sel.cpu().numpy()
    sel_tokens = 0
    G_rows = sel_np.shape[1] // Hkv  # rows per cache head: 1, or G for per-query-head rows
    for i in range(B):
        for h in range(Hkv):  # each (cache head, page) counted once, however many rows select it
            rows = sel_np[i, h * G_rows:(h + 1) * G_rows]
            pages = np.unique(rows[rows >= 0])
            sel_tokens += int(np.minimum(w.page_size, lens[i] - pages * w.page_size).sum())
    kv_bytes = sel_tokens * kv_row * es
    if selector == "coverage":  # the exact page masses: every live key row once
        summ_bytes = int(lens.sum()) * Hkv * D * es
    elif selector == "gaussian":  # the fp32 mean / std rows of every live page
        summ_bytes = int(P.sum()) * Hkv * 2 * D * 4
    score_bytes = summ_bytes + q_bytes
    decode_bytes = kv_bytes + q_bytes + out_bytes
    step_bytes = summ_bytes + kv_bytes + q_bytes + out_bytes
    dense_bytes = int(lens.sum()) * Hkv * kv_row * es + q_bytes + out_bytes
    pk = peaks()
    peak_hbm = pk["hbm"]
    flops_decode = 2 * Hq * (D + w.D_v) * sel_tokens  # QK^T and P.V over the selected tokens
    # the dominant kernel by time (score, select or decode), each timed by its own events
    if t_score >= t_dec and t_score >= t_select:
        # bf16 GQA caches score on the tensor cores (page_score_mma_kernel), fp32 caches on the FMA pipe
        dom = ("mla_qsplit_kernel+mla_score_kernel" if w.latent else
               "page_mass_kernel+coverage_keys_kernel+page_select_kernel" if selector == "coverage" else
               "gauss_score_kernel+page_select_kernel" if selector == "gaussian" else
               "page_score_kernel" if selector == "per-query-head" or w.dtype != "bf16" else "page_score_mma_kernel")
        roof = {"bound": "hbm", "kernel": dom, "achieved": score_bytes / (t_score * 1e-3) / 1e9, "peak": peak_hbm,
                "unit": "GB/s", "algorithmic_per_launch": score_bytes, "algorithmic_unit": "B",
                "launch_us": t_score * 1e3}
    elif w.latent:
        # arithmetic intensity ~300 flop/B, above the measured ridge (~250-290): tensor-bound
        dom = "mla_decode_kernel"
        roof = {"bound": "tensor", "kernel": dom, "achieved": flops_decode / (t_dec * 1e-3) / 1e12,
                "peak": pk["bf16_sustained"], "unit": "TFLOP/s", "algorithmic_per_launch": flops_decode,
                "algorithmic_unit": "flop", "launch_us": t_dec * 1e3,
                "hbm": {"bytes": decode_bytes, "gbs": decode_bytes / (t_dec * 1e-3) / 1e9, "peak": peak_hbm}}
    else:
        dom = "decode_split_kernel"
        roof = {"bound": "hbm", "kernel": dom, "achieved": decode_bytes / (t_dec * 1e-3) / 1e9, "peak": peak_hbm,
                "unit": "GB/s", "algorithmic_per_launch": decode_bytes, "algorithmic_unit": "B",
                "launch_us": t_dec * 1e3}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if args.v_host and dom == "decode_split_kernel":
        roof["note"] = "V of the selected pages crosses NVLink-C2C, not HBM; achieved counts K and V bytes"

    roof["peak_kind"] = pk["kind"] + (" sustained bf16" if roof["bound"] == "tensor" else " copy")
    # the two stages that move the step's bytes, each against its own roofline (`roofline` above is
    # the longer of them); the selection moves no HBM bytes to speak of
    kroof = {"score": {"bound": "hbm", "achieved": score_bytes / (t_score * 1e-3) / 1e9, "peak": peak_hbm,
                       "unit": "GB/s", "launch_us": t_score * 1e3}}
    if w.latent:
        kroof["decode"] = {"bound": "tensor", "achieved": flops_decode / (t_dec * 1e-3) / 1e12,
                           "peak": pk["bf16_sustained"], "unit": "TFLOP/s", "launch_us": t_dec * 1e3}
    else:
        kroof["decode"] = {"bound": "hbm", "achieved": decode_bytes / (t_dec * 1e-3) / 1e9, "peak": peak_hbm,
                           "unit": "GB/s", "launch_us": t_dec * 1e3}
    for kr in kroof.values():
        kr["frac"] = kr["achieved"] / kr["peak"]
    # the captured traffic is of the HBM-resident decode: with V in host memory it does not apply
    # the captured traffic is of the default selector's kernels
    roof["traffic"], scaled = (traffic_of(w.name, dom) if not (args.v_host and dom == "decode_split_kernel")
                               and selector == "bound" else (None, None))
    if scaled:
        roof["traffic_note"] = f"ncu dram read + write per launch, captured on the {scaled}"
    roof["traffic_digest"] = kernel_digest(dom) if dom in KERNEL_SOURCES else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and selector == "bound":
        secs, cores, nseq = oracle_parallel(args.workload, args.batch, 1, args.cpu_seconds)
        cpu = {"value": secs[0] * 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"about {nseq} sequence-steps (in pages) of the {B}-sequence batch through the fp64 oracle's "
                         f"sparse step (score all pages, select, attend), one process per host core for "
                         f"{args.cpu_seconds:.0f} s, scaled to the full batch by pages"}

    clocks = clk.summary()
    graphed = graph_sparse_ms == graph_sparse_ms
    step_ms = graph_sparse_ms if graphed else sparse_ms
    step_dense_ms = graph_dense_ms if graphed else dense_ms
    us = step_ms * 1e3
    line = {
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H_q": Hq, "H_kv": Hkv, "D": D, "page_size": w.page_size,
                   "selector": (selector + (f", coverage {args.coverage} capped at b_max" if selector == "coverage"
                                            else f", z = {args.gauss_z}" if selector == "gaussian" else "")),
                   "contexts": "U[8192, 65536] seeded" if args.workload == 3 else [int(x) for x in lens[:4]],
                   "budget_pages_total": int(w.budgets.sum()),
                   "l2": (f"flushed before every timed step (working set {ws_sparse / 2**20:.0f} MiB sparse, "
                          f"{ws_dense / 2**20:.0f} MiB dense, L2 {l2 / 2**20:.0f} MiB)") if flush else
                         (f"no flush: working set {ws_sparse / 2**20:.0f} MiB sparse, {ws_dense / 2**20:.0f} MiB dense, "
                          f"each over 4x L2 ({l2 / 2**20:.0f} MiB)"),
                   "timing": ("CUDA-graph replay of the step's launches (the append on a second stream beside "
                              "score + select)" if graphed else "eager launches")
                             + "; CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}",
                   "v_cache": ("pinned host memory, read over NVLink-C2C (the selected pages' V bytes do not "
                               "cross HBM; the dense step keeps V in HBM)"
                               + (f"; HBM hot buffer of {hot_pages} (page, head) slots = {args.v_hot:.0%} of each "
                                  "row's selected pages, filled from the warm-up selection the timed steps repeat"
                                  if hot is not None else "")) if args.v_host else "HBM"},
        "roofline": roof,
        "kernels_roofline": kroof,
        "step_hbm": {"bytes": step_bytes, "gbs": step_bytes / (step_ms * 1e-3) / 1e9,
                     "frac_of_measured": step_bytes / (step_ms * 1e-3) / 1e9 / peak_hbm,
                     "frac_of_8TBs": step_bytes / (step_ms * 1e-3) / 1e9 / 8000.0},
        "dense": {"us_per_step": step_dense_ms * 1e3, "bytes": dense_bytes,
                  "gbs": dense_bytes / (step_dense_ms * 1e-3) / 1e9},
        "speedup_vs_dense": step_dense_ms / step_ms,
        "eager": {"us_per_step": sparse_ms * 1e3, "dense_us_per_step": dense_ms * 1e3,
                  "speedup_vs_dense": dense_ms / sparse_ms},
        "kernels_us": {"append": t_app * 1e3, "score": t_score * 1e3, "select": t_select * 1e3,
                       "score_select": (t_score + t_select) * 1e3, "sparse_decode": t_dec * 1e3},
        "score_select_launches": ss_launches,
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "timing": ("CUDA-graph replay" if e2e_ms != e2e_eager_ms else "eager launches")
                          + " of pinned-host H2D copies of q and the new K/V + the step, whose decode writes "
                            "the output straight into a pinned host buffer (the D2H bytes cross NVLink-C2C "
                            "inside the step)",
                "eager_value": e2e_eager_ms * 1e3},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "setup_s": round(setup_s, 1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="psk", choices=["psk", "reference"])
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle window of the cpu_baseline leg")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="--impl reference: total seconds of timed oracle windows over warm-up + steps")
    ap.add_argument("--batch", type=int, default=0, help="use only the first N sequences (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--v-hot", type=float, default=0.0,
                    help="with --v-host: fraction of each row's selected pages kept in an HBM hot buffer")
    ap.add_argument("--v-host", action="store_true",
                    help="keep the value cache in pinned host memory (the value tier; GQA bf16, head_dim 128)")
    ap.add_argument("--selector", default="bound", choices=["bound", "per-query-head", "coverage", "gaussian"],
                    help="the step's page selector: the Quest bound per KV head (default), the bound per "
                         "query head, adaptive coverage over exact page masses (--coverage, capped at the "
                         "workload's b_max), or the Gaussian estimated maximum from mean/std summaries (--gauss-z)")
    ap.add_argument("--coverage", type=float, default=0.95, help="--selector coverage: the mass fraction")
    ap.add_argument("--gauss-z", type=float, default=1.0, help="--selector gaussian: z of mean + z * std")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_psk(args)


if __name__ == "__main__":
    main()
