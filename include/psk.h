/*
 * psk.h -- C ABI of page-selective sparse paged decode attention (one GPU, sm_103a).
 *
 * A decode step has four stages, one call each:
 *
 *   psk_kv_append_and_summarize   write new tokens into the paged K/V cache and keep each
 *                                 page's per-KV-head elementwise key min / max summary
 *                                 in step with it.
 *   psk_page_score_select         score every page with the Quest-style upper bound
 *                                 sum_d max(q_d*kmin_d, q_d*kmax_d), max over the GQA
 *                                 group, times scale; keep the top-b pages per
 *                                 (sequence, KV head) with the sink and tail forced.
 *                                 (_ex: general always-kept sets, budget modes and
 *                                 per-query-head rows; psk_page_score + psk_page_select:
 *                                 the same two stages as separate calls.)
 *   psk_sparse_paged_decode       exact softmax attention over the selected pages only.
 *                                 (_ex: per-query-head rows, value cache in host memory;
 *                                 _noalloc: the same without a caller workspace.)
 *   psk_dense_paged_decode        the same kernel over every page (full-KV baseline).
 *
 * Sources of each operation (pages on page-selective sparse KV attention):
 *   - paged cache [2, num_blocks, page_size, H_kv, D] + block table, per-page key
 *     min/max statistics, attention exact over the selection:
 *     EntmaxKV README (deep-spin/entmaxkv), introduction;
 *   - k_min / k_max refresh on append: EntmaxKV README, kernels/page_metadata.py and the
 *     decode call that appends k_new / v_new (usage example);
 *   - Quest-style page upper bound, top-k with the tail page counted in the budget:
 *     EntmaxKV README, "Two selection strategies", Top-k; kernels/page_criticality.py,
 *     kernels/page_topk.py;
 *   - static top-b per (layer, KV head), sink and recent pages always kept and counted
 *     inside b, GQA group combined by max: LOCKS (locks-kv) PKG-INFO, "How it works",
 *     "Results" preamble and the configuration table (sink_pages / window_pages = 1 / 1,
 *     quad_combine = max);
 *   - prefill untouched, sparse decode reads only the selected pages: LOCKS PKG-INFO,
 *     "How it works", Sparse decode; AMASS (amass-kv) PyPI page, introduction.
 *
 * Conventions for every call
 *   - All tensor pointers address contiguous memory in the layouts stated, 16-byte aligned.
 *     k_cache, summaries, the workspace, v_cache (unless PSK_DECODE_V_HOST) and the latent
 *     form's q are read by TMA / bulk copies or atomics and must be device memory; the other
 *     buffers (q, k_new, v_new, block_table, seq_lens, budgets, selected, scores_out, out)
 *     may also be host memory the GPU addresses directly (pinned, under unified addressing),
 *     e.g. an output written straight to the host. Index tensors are int32. q, k_new, v_new,
 *     caches, summaries and out share the storage type `layout->dtype` (PSK_BF16 or
 *     PSK_F32); arithmetic is fp32. With PSK_BF16 the page scores and q.k products run on the
 *     tensor cores (bf16 x bf16 products are exact in fp32, sums are fp32), and the decode's
 *     softmax weights enter P.V as the sum of two bf16 values (about 16 significant bits).
 *   - The caller owns every buffer. The library allocates nothing, frees nothing and
 *     keeps no state between calls apart from what it writes into the caller's buffers.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream). Host-side argument checks happen before any launch and are synchronous.
 *   - Kernels are launched with programmatic stream serialisation (programmatic dependent
 *     launch): a kernel may be scheduled while the kernel before it on `stream` drains, but
 *     it waits for that kernel's completion (griddepcontrol.wait) before it reads or writes
 *     any global memory, so stream order is kept exactly. Setting PSK_PDL=0 in the
 *     environment before the first call launches in plain stream order.
 *   - Return value: PSK_OK or a psk_status code. PSK_ERR_CUDA reports a launch error.
 *   - Device-side violations that the host cannot see (a block id outside
 *     [0, num_blocks), a sequence longer than max_pages pages, a bad selected id, a
 *     budget below the always-kept page count) set a sticky bit in the workspace status
 *     word and skip the affected unit (its selected row is written as -1, its output
 *     rows as zeros); read it with psk_get_device_status. Nothing traps, asserts or waits.
 *   - Workspace: every call takes a caller-allocated workspace of at least the size the
 *     matching psk_*_workspace_size query returns; one buffer sized for the largest may
 *     be shared by all calls on one stream. It must be zero-filled once before its first
 *     use (every call leaves its internal counters at zero again); the status word stays
 *     set until psk_clear_device_status. Calls sharing one workspace must not overlap on
 *     the GPU (use one stream, or one workspace per stream).
 *   - Preconditions the library does not check: no two live logical pages map to the same
 *     physical block; inputs are finite.
 */
#ifndef PSK_H
#define PSK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *psk_stream_t; /* a cudaStream_t */

enum psk_dtype { PSK_F32 = 0, PSK_BF16 = 1 };

enum psk_status {
  PSK_OK = 0,
  PSK_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, inconsistent shape       */
  PSK_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, page_size, group size, ... */
  PSK_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the size query returns  */
  PSK_ERR_CUDA = 4         /* a CUDA launch failed (cudaGetLastError after the launch)  */
};

/* sticky device status bits (psk_get_device_status) */
#define PSK_DEV_BAD_BLOCK 0x1u    /* block-table entry outside [0, num_blocks)              */
#define PSK_DEV_BAD_SEQLEN 0x2u   /* seq_len < 1, or more than max_pages pages              */
#define PSK_DEV_BAD_SELECTED 0x4u /* selected id outside [0, P) or list not ascending       */
#define PSK_DEV_BAD_BUDGET 0x8u   /* budget below the always-kept count, or above b_max      */
#define PSK_DEV_BAD_APPEND 0x10u  /* append position outside the block-table row, or n < 0  */
#define PSK_DEV_TIMEOUT 0x20u     /* a bounded wait for an asynchronous copy gave up         */

/*
 * Geometry of one layer's paged cache and of the decode batch.
 *
 *   k_cache  [num_blocks, page_size, num_kv_heads, head_dim]      (the K half of vLLM's
 *   v_cache  [num_blocks, page_size, num_kv_heads, v_head_dim]     [2, num_blocks, ...])
 *   summaries[num_blocks, num_kv_heads, 2, head_dim]  kmin at [...,0,:], kmax at [...,1,:],
 *             indexed by PHYSICAL block, storage dtype (min / max are exact in any dtype)
 *   block_table [batch, max_pages] int32: logical page -> physical block
 *   seq_lens    [batch] int32 (tokens in the cache, >= 1)
 *   q           [batch, num_q_heads, head_dim]; query head g reads KV head
 *               g / (num_q_heads / num_kv_heads)
 *   out         [batch, num_q_heads, v_head_dim]
 *
 * latent = 1 selects the MLA form: num_kv_heads = 1, the cache holds one latent vector per
 * token (k_cache), the value is its first v_head_dim elements and v_cache must be NULL.
 *
 * Selection limit: a sequence longer than one selection chunk (4096, 8192 or 16384 pages) is
 * selected chunk by chunk and the chunks' winners are merged by one CTA holding at most 8192
 * candidates, so score / select calls need some chunk c in {4096, 8192, 16384} with
 * ceil(max_pages / c) = 1 or ceil(max_pages / c) * min(b_max - 1, c) <= 8192 (e.g. max_pages =
 * 65536 allows b_max up to 2049); otherwise they return PSK_ERR_UNSUPPORTED (size query: 0).
 *
 * Built shapes (anything else returns PSK_ERR_UNSUPPORTED and a workspace size of 0):
 *   GQA: v_head_dim = head_dim; page_size 16, 32, 48 or 64; num_kv_heads a divisor or a
 *        multiple of 8; PSK_BF16 with head_dim 64 or 128 and group size
 *        G = num_q_heads / num_kv_heads of 1, 2 or 4, and G = 8 at head_dim 128 (score, select
 *        and decode; the coverage and Gaussian calls take G of 1, 2 or 4); PSK_F32 with head_dim
 *        64 or 128 and G of 1 or 4.
 *   MLA: PSK_BF16, num_q_heads 128, head_dim 576, v_head_dim 512, page_size 32 or 64.
 */
typedef struct psk_layout {
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t v_head_dim;
  int32_t page_size;
  int32_t num_blocks;
  int32_t max_pages;
  int32_t dtype; /* enum psk_dtype */
  int32_t latent;
} psk_layout;

/* ---------------------------------------------------------------------------------------
 * Stage 1: append tokens and refresh page summaries.
 *
 * For sequence i, the n_i = cu_new[i+1] - cu_new[i] rows k_new[cu_new[i] + j] (j < n_i)
 * are written at token positions t = start_pos[i] + j: slot t % page_size of physical block
 * block_table[i][t / page_size]. Every page the call touches gets its summary refreshed so
 * that it covers all tokens of the page below start_pos[i] + n_i: a page whose first token
 * is written by this call starts a fresh summary; a page that already held tokens is widened
 * by the new ones (elementwise min / max, -0.0 ordered below +0.0).
 *   decode: n_i = 1, start_pos = the sequence length before the append;
 *   prefill: start_pos = 0, n_i = prompt length.
 * seq_lens is NOT modified: after the call the caller's length is start_pos[i] + n_i.
 *
 *   k_new [total_new, num_kv_heads, head_dim], v_new [total_new, num_kv_heads, v_head_dim]
 *   (latent: v_new and v_cache NULL). start_pos [batch], cu_new [batch + 1] device int32.
 *   total_new = cu_new[batch]; max_new >= every n_i (sizes the launch grid).
 * --------------------------------------------------------------------------------------- */
int psk_kv_append_and_summarize(const psk_layout *layout, const void *k_new, const void *v_new,
                                const int32_t *start_pos, const int32_t *cu_new, int32_t total_new,
                                int32_t max_new, void *k_cache, void *v_cache, void *summaries,
                                const int32_t *block_table, void *workspace, size_t workspace_bytes,
                                psk_stream_t stream);

/* The same with an optional second summary store (EntmaxKV README, introduction: pages are
 * scored from per-page key statistics, "mean/std for Gaussian"; repository layout,
 * gaussian/page_metadata.py, "Per-page k_mean / k_std refresh"):
 *   stats  fp32 [num_blocks, num_kv_heads, 2, head_dim], device memory, indexed by physical
 *          block: the elementwise mean of the page's valid keys at [...,0,:] and their population
 *          standard deviation (divisor = the page's token count) at [...,1,:].
 * Every page the call touches gets both recomputed in fp32 from all of its tokens below
 * start_pos[i] + n_i (two passes over the page's rows in the cache), so they never drift from a
 * rebuild. summaries or stats may be NULL (not both); psk_kv_append_and_summarize is this call
 * with stats = NULL. */
int psk_kv_append_and_summarize_ex(const psk_layout *layout, const void *k_new, const void *v_new,
                                   const int32_t *start_pos, const int32_t *cu_new, int32_t total_new,
                                   int32_t max_new, void *k_cache, void *v_cache, void *summaries,
                                   float *stats, const int32_t *block_table, void *workspace,
                                   size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stages 2 + 3: page scores and top-b selection.
 *
 * For sequence i with P_i = ceil(seq_lens[i] / page_size) pages and KV head h:
 *   score[i,h,p] = scale * max_{g in group(h)} sum_d max(q[i,g,d]*kmin[p,h,d], q[i,g,d]*kmax[p,h,d])
 * with the summaries of block block_table[i][p]. Selected pages: the sink 0 and the tail
 * P_i - 1 always, plus the min(b_i, P_i) - |{0, P_i - 1}| highest-scoring other pages, ties
 * to the lower page index. b_i = budgets[i] (int32 [batch], 2 <= b_i <= b_max, or any
 * 1 <= b_i <= b_max when P_i == 1).
 *
 *   selected  [batch, num_kv_heads, b_max] int32 out: ascending logical page ids, padded
 *             with -1 after the min(b_i, P_i) valid entries.
 *   scores_out [batch, num_kv_heads, max_pages] fp32 out, optional (NULL = not written):
 *             the scores above for p < P_i; entries p >= P_i are left untouched.
 * Scores accumulate in fp32. scale is normally 1/sqrt(head_dim).
 * Without scores_out the summaries of the sink and the tail page are not read (those pages
 * are kept whatever their score), so a one-token decode append, which touches only the tail
 * page, may run concurrently with this call on another stream.
 * --------------------------------------------------------------------------------------- */
int psk_page_score_select(const psk_layout *layout, const void *q, const void *summaries,
                          const int32_t *block_table, const int32_t *seq_lens,
                          const int32_t *budgets, int32_t b_max, float scale, int32_t *selected,
                          float *scores_out, void *workspace, size_t workspace_bytes,
                          psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stages 2 + 3 with general always-kept sets and budget modes (LOCKS PKG-INFO,
 * "Configuration (LocksConfig)": sink_pages / window_pages, budget, budget_pages).
 *
 * Always-kept pages of sequence i: F_i = [0, sink_pages) U [P_i - window_pages, P_i), clipped
 * to [0, P_i); |F_i| = min(P_i, sink_pages + window_pages); sink_pages >= 0, window_pages >= 1
 * (the tail page is always kept). The budget b_i counts them:
 *   PSK_BUDGET_PER_SEQUENCE  b_i = budgets[i] (device int32 [batch]); a b_i below |F_i| or
 *                            above b_max flags PSK_DEV_BAD_BUDGET and writes the row as -1;
 *   PSK_BUDGET_PAGES         b_i = max(|F_i|, min(P_i, budget_pages)), budget_pages >= 1;
 *   PSK_BUDGET_FRACTION      b_i = max(|F_i|, min(P_i, max(1, ceil(P_i * budget_fraction)))),
 *                            0 < budget_fraction <= 1, P_i * budget_fraction evaluated in IEEE
 *                            double (the retained-count rule of the vllm-rlt pull request #157
 *                            discussion: a ceiling, not rounding to nearest).
 * Selected: F_i plus the min(b_i, P_i) - |F_i| highest-scoring other pages, ties to the lower
 * page index, ascending, padded with -1 to b_max. For the two scalar modes the call returns
 * PSK_ERR_INVALID_ARG unless b_max holds the largest b_i any sequence of at most max_pages
 * pages can get. Everything else is as psk_page_score_select, which is this call with
 * PSK_BUDGET_PER_SEQUENCE and sink_pages = window_pages = 1. Without scores_out the
 * summaries of the always-kept pages are not read.
 *
 * per_query_head = 1 (GQA only; EntmaxKV README, "Two selection strategies", Top-k: pages are
 * kept per query head) ranks and selects pages for every query head g on its own, with
 *   score[i,g,p] = scale * sum_d max(q[i,g,d]*kmin[p,h,d], q[i,g,d]*kmax[p,h,d]),  h = g / G,
 * so selected is [batch, num_q_heads, b_max] and scores_out [batch, num_q_heads, max_pages];
 * decode such rows with psk_sparse_paged_decode_ex and PSK_DECODE_PER_QUERY_HEAD. Each query
 * head then reads its own pages, so the decode moves up to G times the K/V bytes of per-KV-head
 * selection at the same budget.
 * --------------------------------------------------------------------------------------- */
enum psk_budget_mode { PSK_BUDGET_PER_SEQUENCE = 0, PSK_BUDGET_PAGES = 1, PSK_BUDGET_FRACTION = 2 };

typedef struct psk_select_params {
  const int32_t *budgets;  /* PSK_BUDGET_PER_SEQUENCE: device int32 [batch]; else ignored */
  double budget_fraction;  /* PSK_BUDGET_FRACTION                                         */
  int32_t budget_pages;    /* PSK_BUDGET_PAGES                                            */
  int32_t mode;            /* enum psk_budget_mode                                        */
  int32_t sink_pages;      /* >= 0                                                        */
  int32_t window_pages;    /* >= 1                                                        */
  int32_t per_query_head;  /* 0: one row per (sequence, KV head); 1: per (sequence, q head) */
} psk_select_params;

int psk_page_score_select_ex(const psk_layout *layout, const void *q, const void *summaries,
                             const int32_t *block_table, const int32_t *seq_lens,
                             const psk_select_params *params, int32_t b_max, float scale,
                             int32_t *selected, float *scores_out, void *workspace,
                             size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stages 2 + 3 with the Gaussian page score instead of the bound (EntmaxKV README, "Two
 * selection strategies", Gaussian-aware: each page's scores modelled as a Gaussian, pages kept
 * whose estimated maximum is high). From the mean / std store of psk_kv_append_and_summarize_ex:
 *   score[i,h,p] = scale * max_{g in group(h)} (q[i,g] . mean[p,h]
 *                                                + z * sqrt(sum_d (q[i,g,d] * std[p,h,d])^2)),
 * i.e. the page's logits modelled as a Gaussian with independent dimensions and its maximum
 * estimated as mean + z standard deviations (z chosen by the caller, e.g. 1.5 to 2.5 for 16-
 * token pages). The top-b pages are then selected exactly as psk_page_score_select_ex does
 * (params: budget modes, sink / window pages; per_query_head must be 0). GQA only (head_dim 64
 * or 128). The threshold solve of the entmax normaliser that the Gaussian selector uses is not
 * part of this library: pages are ranked by the estimated maximum and the budget decides how
 * many are kept. Same workspace as psk_page_score_select_ex.
 * --------------------------------------------------------------------------------------- */
int psk_page_score_select_gaussian(const psk_layout *layout, const void *q, const float *stats,
                                   const int32_t *block_table, const int32_t *seq_lens,
                                   const psk_select_params *params, int32_t b_max, float scale,
                                   float z, int32_t *selected, float *scores_out, void *workspace,
                                   size_t workspace_bytes, psk_stream_t stream);

/* Kernel launches one psk_page_score_select_ex call makes for this layout, b_max and
 * per_query_head (0 when the layout is invalid or unsupported): 2 for GQA caches (score,
 * selection), 3 for the latent form (query split, score, selection). Useful for sizing CUDA
 * graphs and counting launches. */
int psk_score_select_launches(const psk_layout *layout, int32_t b_max, int32_t per_query_head);

/* ---------------------------------------------------------------------------------------
 * Stages 2 + 3 in the adaptive coverage mode (LOCKS PKG-INFO, "Configuration (LocksConfig)",
 * `coverage`: adaptive per-head nucleus coverage over exact page masses, GQA only; AMASS PyPI
 * page, "Key AmassConfig fields", the same option). Instead of a bound from the summaries,
 * every page's exact softmax mass is computed from the keys themselves (a K-only pass over
 * every page):
 *   mass[i,g,p] = sum over tokens t of page p (t < seq_lens[i]) of softmax_t(scale * q[i,g] . k_t),
 * the softmax over every token of sequence i in KV head h = g / G; the unit (i, h) takes
 * mass[i,h,p] = max over the group's query heads. Selected: the always-kept pages
 * [0, sink_pages) U [P_i - window_pages, P_i), then the other pages in order of mass (desc,
 * ties to the lower page) until the selected mass reaches coverage times the unit's total mass
 * (0 < coverage <= 1), at most b_max pages in all. Rows as psk_page_score_select:
 * selected [batch, num_kv_heads, b_max] ascending, -1 padded. masses_out (optional, fp32
 * [batch, num_kv_heads, max_pages]) receives mass[i,h,p] for p < P_i. Masses are fp32; their
 * sums are taken in fixed point (units of 2^-40), so the selection does not depend on
 * summation order. Reads k_cache (device memory) for every page, i.e. half the bytes of a
 * dense decode. The workspace is the one psk_coverage_workspace_size reports.
 * --------------------------------------------------------------------------------------- */
int psk_page_select_coverage(const psk_layout *layout, const void *q, const void *k_cache,
                             const int32_t *block_table, const int32_t *seq_lens, double coverage,
                             int32_t sink_pages, int32_t window_pages, int32_t b_max, float scale,
                             int32_t *selected, float *masses_out, void *workspace,
                             size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * The two stages of psk_page_score_select_ex as separate calls, for callers that run other
 * work between them or time them apart. psk_page_score writes one selection key per
 * (unit, page) into the workspace (and scores_out when given); psk_page_select turns those
 * keys into the selected rows. The pair must be made in that order on one stream with the
 * same workspace, layout, params and b_max, and no other call on that workspace in between
 * (the keys live in its per-call scratch). Their results equal psk_page_score_select_ex's.
 * psk_page_select reads seq_lens, the budget and the always-kept sizes from params, and the keys.
 * --------------------------------------------------------------------------------------- */
int psk_page_score(const psk_layout *layout, const void *q, const void *summaries,
                   const int32_t *block_table, const int32_t *seq_lens,
                   const psk_select_params *params, int32_t b_max, float scale, float *scores_out,
                   void *workspace, size_t workspace_bytes, psk_stream_t stream);
int psk_page_select(const psk_layout *layout, const int32_t *seq_lens,
                    const psk_select_params *params, int32_t b_max, int32_t *selected,
                    void *workspace, size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stage 4: exact softmax attention over the selected pages.
 *
 *   out[i,g,:] = sum_t softmax_t(scale * q[i,g] . k_t) v_t
 * over the tokens t < seq_lens[i] of the pages listed in selected[i, g / G, :] (read up to
 * the first -1 or b_max entries; ids must be ascending and in [0, P_i)). The pages are split
 * across CTAs; each split keeps an fp32 online-softmax state (m, l, O) and a combine pass
 * merges the splits by log-sum-exp. out is written in the storage dtype.
 * --------------------------------------------------------------------------------------- */
int psk_sparse_paged_decode(const psk_layout *layout, const void *q, const void *k_cache,
                            const void *v_cache, const int32_t *block_table,
                            const int32_t *seq_lens, const int32_t *selected, int32_t b_max,
                            float scale, void *out, void *workspace, size_t workspace_bytes,
                            psk_stream_t stream);

/* Full-KV decode with the same kernel skeleton: every page 0 .. P_i - 1 of every KV head. */
int psk_dense_paged_decode(const psk_layout *layout, const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *block_table,
                           const int32_t *seq_lens, float scale, void *out, void *workspace,
                           size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * psk_sparse_paged_decode with flags (below). PSK_DECODE_PER_QUERY_HEAD: selected is
 * [batch, num_q_heads, b_max] (rows of psk_page_score_select_ex with per_query_head = 1) and
 * query head g attends its own row's pages of KV head g / G. flags = 0 is
 * psk_sparse_paged_decode. GQA only; the workspace is the one psk_sparse_decode_workspace_size
 * sizes (it covers both forms).
 * --------------------------------------------------------------------------------------- */
#define PSK_DECODE_PER_QUERY_HEAD 0x1u
/* PSK_DECODE_V_HOST: the value tier in host memory (LOCKS PKG-INFO, "Configuration", variant
 * mem-v: V in DRAM, K resident). v_cache is host memory the GPU can address directly (pinned
 * with cudaHostAlloc / cudaMallocHost, addressed by its host pointer under unified addressing)
 * and is read over NVLink-C2C with plain loads, only for the selected pages' valid rows; K, the
 * summaries and the rest stay in device memory. psk_kv_append_and_summarize writes new values
 * to such a v_cache directly. Built for sparse GQA decode, PSK_BF16, head_dim 128 (else
 * PSK_ERR_UNSUPPORTED). */
#define PSK_DECODE_V_HOST 0x2u
int psk_sparse_paged_decode_ex(const psk_layout *layout, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_table,
                               const int32_t *seq_lens, const int32_t *selected, int32_t b_max,
                               float scale, uint32_t flags, void *out, void *workspace,
                               size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * The value tier with a resident hot buffer (LOCKS PKG-INFO, "How it works", Optional DRAM tier
 * (Stage B): V in a pinned host pool, the pages called each step resident; AMASS PyPI page: a
 * pinned, device-mapped host pool with a bounded resident hot buffer plus staging).
 *
 *   v_hot   device bf16 [n_slots, page_size, v_head_dim]: slot s holds one KV head's V rows of
 *           one page.
 *   v_slot  device int32 [batch, num_kv_heads, max_pages]: the slot holding (sequence, KV head,
 *           logical page), or -1. The caller owns the map and the replacement policy (for
 *           example, keep the pages selected on the previous steps) and changes it only through
 *           psk_value_tier_fill (or its own copies, in stream order with the decode).
 *
 * psk_sparse_paged_decode_tiered is psk_sparse_paged_decode_ex with PSK_DECODE_V_HOST, except
 * that a selected page with a slot is read from v_hot (HBM) instead of over NVLink-C2C. The tail
 * page P_i - 1 is always read from the host cache (it still takes appends); full pages never
 * change, so their resident copies stay exact. A slot >= n_slots flags PSK_DEV_BAD_SELECTED and
 * the page is read from the host. Results are bit-identical to the device-memory decode.
 * PSK_BF16, GQA, head_dim 128.
 *
 * psk_value_tier_fill runs n_entries fill / evict steps, entries int32 [n_entries, 4] (device):
 * (sequence, KV head, logical page, slot). slot >= 0 copies the page's page_size V rows of that
 * head from the host cache into v_hot[slot] and sets v_slot for it; slot < 0 sets v_slot to -1.
 * Entries must not name the same slot or the same (sequence, head, page) twice. Out-of-range
 * entries flag PSK_DEV_BAD_SELECTED, bad block ids PSK_DEV_BAD_BLOCK, and are skipped. The
 * workspace is only used for the status word.
 * --------------------------------------------------------------------------------------- */
int psk_sparse_paged_decode_tiered(const psk_layout *layout, const void *q, const void *k_cache,
                                   const void *v_cache_host, const void *v_hot, int32_t n_slots,
                                   const int32_t *v_slot, const int32_t *block_table,
                                   const int32_t *seq_lens, const int32_t *selected, int32_t b_max,
                                   float scale, void *out, void *workspace, size_t workspace_bytes,
                                   psk_stream_t stream);
int psk_value_tier_fill(const psk_layout *layout, const void *v_cache_host,
                        const int32_t *block_table, const int32_t *entries, int32_t n_entries,
                        void *v_hot, int32_t n_slots, int32_t *v_slot, void *workspace,
                        size_t workspace_bytes, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stage 4 without a workspace (no counterpart in the pages: an addition for callers that
 * cannot allocate device memory). Some host programs own every byte of device memory
 * through their own allocator and pass a plugin only its inputs and outputs, or run a loop
 * that must never call cudaMalloc. This call computes what psk_sparse_paged_decode computes
 * for the GQA form (rows per (sequence, KV head), values in device memory; no _ex flags;
 * latent layouts return PSK_ERR_UNSUPPORTED), but keeps its split partials in a 32 MiB
 * device array inside the library (one per GPU, held until exit); it allocates nothing.
 *   - Returns PSK_ERR_WORKSPACE when the partials (the size psk_sparse_decode_workspace_size
 *     reports) exceed 32 MiB.
 *   - Each call looks up the array's address in the current context (cudaGetSymbolAddress).
 *     With lazy module loading (the CUDA default) the first call on each device loads the
 *     array, which may synchronise: make one warm-up call before any stream capture or
 *     latency-critical loop, or set CUDA_MODULE_LOADING=EAGER.
 *   - All calls share the one array: calls that overlap on the GPU race and must be
 *     serialised by the caller. Each call zeroes the array's header before use.
 *   - Device-side input violations are not reported (the status word is internal).
 * --------------------------------------------------------------------------------------- */
int psk_sparse_paged_decode_noalloc(const psk_layout *layout, const void *q, const void *k_cache,
                                    const void *v_cache, const int32_t *block_table,
                                    const int32_t *seq_lens, const int32_t *selected, int32_t b_max,
                                    float scale, void *out, psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Self-test of the bounded waits (failure detection; no counterpart in the pages). Every
 * streaming kernel waits for its asynchronous copies on mbarriers with a bounded number of
 * polls and, if a copy never lands, sets PSK_DEV_TIMEOUT and returns instead of hanging. This
 * call runs that same wait, with spin_limit polls (1 .. 4194304, the kernels' own limit), on a
 * phase that cannot complete (an expected transaction count with no copy issued), so the
 * timeout path can be observed: afterwards psk_get_device_status reports PSK_DEV_TIMEOUT and
 * the context stays usable (nothing was in flight). Asynchronous on `stream`.
 * --------------------------------------------------------------------------------------- */
int psk_selftest_bounded_wait(void *workspace, size_t workspace_bytes, uint32_t spin_limit,
                              psk_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Workspace sizes (bytes). Return 0 when the layout is invalid or unsupported.
 * --------------------------------------------------------------------------------------- */
size_t psk_append_workspace_size(const psk_layout *layout);
size_t psk_score_select_workspace_size(const psk_layout *layout, int32_t b_max);
size_t psk_sparse_decode_workspace_size(const psk_layout *layout, int32_t b_max);
size_t psk_dense_decode_workspace_size(const psk_layout *layout);
size_t psk_coverage_workspace_size(const psk_layout *layout, int32_t b_max);

/* Copy the sticky device status word of `workspace` to *flags (synchronises `stream`). */
int psk_get_device_status(const void *workspace, uint32_t *flags, psk_stream_t stream);
/* Zero the status word (asynchronous on `stream`). */
int psk_clear_device_status(void *workspace, psk_stream_t stream);

/* Short English description of a psk_status code (static storage). */
const char *psk_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int psk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PSK_H */
