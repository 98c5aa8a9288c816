// C ABI of libpsk: host-side argument checks, workspace planning and kernel dispatch.
// Every entry point validates before it launches anything and never allocates.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "psk_common.cuh"
#include "psk_internal.h"

using namespace psk;

namespace {

int elem_bytes(int dtype) { return dtype == PSK_F32 ? 4 : 2; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every call.
int check_layout(const psk_layout *L) {
  if (!L) return PSK_ERR_INVALID_ARG;
  if (L->batch < 1 || L->num_q_heads < 1 || L->num_kv_heads < 1 || L->head_dim < 1 || L->v_head_dim < 1 ||
      L->page_size < 1 || L->num_blocks < 1 || L->max_pages < 1)
    return PSK_ERR_INVALID_ARG;
  if (L->num_q_heads % L->num_kv_heads != 0) return PSK_ERR_INVALID_ARG;
  if (L->dtype != PSK_F32 && L->dtype != PSK_BF16) return PSK_ERR_INVALID_ARG;
  if (L->latent != 0 && L->latent != 1) return PSK_ERR_INVALID_ARG;
  if (L->latent && (L->num_kv_heads != 1 || L->v_head_dim > L->head_dim)) return PSK_ERR_INVALID_ARG;
  const int es = elem_bytes(L->dtype);
  if ((L->head_dim * es) % 16 != 0 || (L->v_head_dim * es) % 16 != 0) return PSK_ERR_UNSUPPORTED;
  return PSK_OK;
}

int check_gqa_compute(const psk_layout *L) {
  if (L->latent) return mla_supported(*L) ? PSK_OK : PSK_ERR_UNSUPPORTED;
  const int G = L->num_q_heads / L->num_kv_heads;
  if (!score_supported(L->dtype, L->head_dim, G)) return PSK_ERR_UNSUPPORTED;
  if (!decode_supported(L->dtype, L->head_dim, L->v_head_dim, G, L->page_size)) return PSK_ERR_UNSUPPORTED;
  return PSK_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PSK_OK : PSK_ERR_CUDA; }

// The per-query-head view of a GQA layout: one unit head per query head (num_kv_heads =
// num_q_heads, group size 1); unit head h reads cache head h >> kv_shift, G = 2^kv_shift. False
// when that form is not built for this layout (G not a power of two included).
bool per_query_head_view(const psk_layout &L, psk_layout *V, int *kv_shift) {
  if (L.latent) return false;
  const int G = L.num_q_heads / L.num_kv_heads;
  if (G & (G - 1)) return false;
  *V = L;
  V->num_kv_heads = L.num_q_heads;
  *kv_shift = __builtin_ctz((unsigned)G);
  return score_supported(L.dtype, L.head_dim, 1) &&
         decode_supported(L.dtype, L.head_dim, L.v_head_dim, 1, L.page_size);
}

}  // namespace

extern "C" {

int psk_version(void) { return 100; }

const char *psk_status_string(int status) {
  switch (status) {
    case PSK_OK: return "ok";
    case PSK_ERR_INVALID_ARG: return "invalid argument";
    case PSK_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PSK_ERR_WORKSPACE: return "workspace missing or too small";
    case PSK_ERR_CUDA: return "CUDA launch error";
    default: return "unknown status";
  }
}

size_t psk_append_workspace_size(const psk_layout *layout) {
  return check_layout(layout) == PSK_OK ? kWsHeader : 0;
}

// Score / select and sparse decode sizes cover both the per-KV-head and the per-query-head
// forms, so one workspace serves every call of a layout.
size_t psk_score_select_workspace_size(const psk_layout *layout, int32_t b_max) {
  if (check_layout(layout) != PSK_OK || check_gqa_compute(layout) != PSK_OK || b_max < 1) return 0;
  ScorePlan plan;
  if (!plan_score(*layout, b_max, &plan)) return 0;
  size_t bytes = plan.ws_bytes;
  psk_layout V;
  int kv_shift;
  if (per_query_head_view(*layout, &V, &kv_shift) && plan_score(V, b_max, &plan, kv_shift))
    bytes = std::max(bytes, plan.ws_bytes);
  return bytes;
}

int psk_score_select_launches(const psk_layout *layout, int32_t b_max, int32_t per_query_head) {
  if (check_layout(layout) != PSK_OK || check_gqa_compute(layout) != PSK_OK || b_max < 1) return 0;
  if (per_query_head != 0 && per_query_head != 1) return 0;
  psk_layout U = *layout;
  int kv_shift = 0;
  if (per_query_head && !per_query_head_view(*layout, &U, &kv_shift)) return 0;
  ScorePlan plan;
  if (!plan_score(U, b_max, &plan, kv_shift)) return 0;
  return layout->latent ? 3 : 2;
}

static bool plan_any_decode(const psk_layout &L, int entries, bool dense, DecodePlan *plan) {
  return L.latent ? plan_mla_decode(L, entries, plan) : plan_decode(L, entries, dense, plan);
}

size_t psk_sparse_decode_workspace_size(const psk_layout *layout, int32_t b_max) {
  if (check_layout(layout) != PSK_OK || check_gqa_compute(layout) != PSK_OK || b_max < 1) return 0;
  DecodePlan plan;
  if (!plan_any_decode(*layout, b_max, false, &plan)) return 0;
  size_t bytes = plan.ws_bytes;
  psk_layout V;
  int kv_shift;
  if (per_query_head_view(*layout, &V, &kv_shift) && plan_decode(V, b_max, false, &plan))
    bytes = std::max(bytes, plan.ws_bytes);
  return bytes;
}

size_t psk_dense_decode_workspace_size(const psk_layout *layout) {
  if (check_layout(layout) != PSK_OK || check_gqa_compute(layout) != PSK_OK) return 0;
  DecodePlan plan;
  return plan_any_decode(*layout, layout->max_pages, true, &plan) ? plan.ws_bytes : 0;
}

int psk_get_device_status(const void *workspace, uint32_t *flags, psk_stream_t stream) {
  if (!workspace || !flags) return PSK_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return PSK_ERR_CUDA;
  *flags = v;
  return PSK_OK;
}

int psk_clear_device_status(void *workspace, psk_stream_t stream) {
  if (!workspace) return PSK_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)));
}

int psk_kv_append_and_summarize_ex(const psk_layout *layout, const void *k_new, const void *v_new,
                                   const int32_t *start_pos, const int32_t *cu_new, int32_t total_new,
                                   int32_t max_new, void *k_cache, void *v_cache, void *summaries, float *stats,
                                   const int32_t *block_table, void *workspace, size_t workspace_bytes,
                                   psk_stream_t stream) {
  int rc = check_layout(layout);
  if (rc != PSK_OK) return rc;
  const psk_layout &L = *layout;
  if (total_new < 0 || max_new < 0) return PSK_ERR_INVALID_ARG;
  if (!start_pos || !cu_new || !k_cache || !block_table || (!summaries && !stats)) return PSK_ERR_INVALID_ARG;
  if (L.latent ? (v_new != nullptr || v_cache != nullptr) : (!v_cache || (total_new > 0 && !v_new)))
    return PSK_ERR_INVALID_ARG;
  if (total_new > 0 && !k_new) return PSK_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(summaries) || !aligned16(stats))
    return PSK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWsHeader) return PSK_ERR_WORKSPACE;
  if (total_new == 0 || max_new == 0) return PSK_OK;
  AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.start_pos = start_pos;
  a.cu_new = cu_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.summaries = summaries;
  a.stats = stats;
  a.block_table = block_table;
  a.ws = workspace;
  a.B = L.batch;
  a.H_kv = L.num_kv_heads;
  a.D = L.head_dim;
  a.D_v = L.v_head_dim;
  a.ps = L.page_size;
  a.nb = L.num_blocks;
  a.max_pages = L.max_pages;
  return cuda_status(launch_append(a, L.dtype, max_new, static_cast<cudaStream_t>(stream)));
}

int psk_kv_append_and_summarize(const psk_layout *layout, const void *k_new, const void *v_new,
                                const int32_t *start_pos, const int32_t *cu_new, int32_t total_new,
                                int32_t max_new, void *k_cache, void *v_cache, void *summaries,
                                const int32_t *block_table, void *workspace, size_t workspace_bytes,
                                psk_stream_t stream) {
  if (!summaries) return PSK_ERR_INVALID_ARG;
  return psk_kv_append_and_summarize_ex(layout, k_new, v_new, start_pos, cu_new, total_new, max_new, k_cache, v_cache,
                                        summaries, nullptr, block_table, workspace, workspace_bytes, stream);
}

int psk_page_score_select(const psk_layout *layout, const void *q, const void *summaries,
                          const int32_t *block_table, const int32_t *seq_lens, const int32_t *budgets,
                          int32_t b_max, float scale, int32_t *selected, float *scores_out, void *workspace,
                          size_t workspace_bytes, psk_stream_t stream) {
  psk_select_params params = {};
  params.budgets = budgets;
  params.mode = PSK_BUDGET_PER_SEQUENCE;
  params.sink_pages = 1;
  params.window_pages = 1;
  return psk_page_score_select_ex(layout, q, summaries, block_table, seq_lens, &params, b_max, scale, selected,
                                  scores_out, workspace, workspace_bytes, stream);
}

// Largest budget a sequence of P pages gets in a scalar budget mode (the same arithmetic as
// the select kernel's).
static long long scalar_mode_budget(const psk_select_params &sp, long long P) {
  const long long forced = std::min(P, (long long)sp.sink_pages + sp.window_pages);
  long long b;
  if (sp.mode == PSK_BUDGET_FRACTION)
    b = std::min(P, std::max(1LL, (long long)std::ceil((double)P * sp.budget_fraction)));
  else
    b = std::min(P, (long long)sp.budget_pages);
  return std::max(forced, b);
}

// Score and / or select (stages: kStageScore, kStageSelect). A select-only call reads the keys
// a score-only call left in the same workspace.
static int score_select_common(const psk_layout *layout, const void *q, const void *summaries,
                               const int32_t *block_table, const int32_t *seq_lens, const psk_select_params *params,
                               int32_t b_max, float scale, int32_t *selected, float *scores_out, void *workspace,
                               size_t workspace_bytes, psk_stream_t stream, int stages, const float *gauss_stats = nullptr,
                               float gauss_z = 0.f) {
  int rc = check_layout(layout);
  if (rc != PSK_OK) return rc;
  const psk_layout &L = *layout;
  const bool do_score = (stages & kStageScore) != 0, do_select = (stages & kStageSelect) != 0;
  if (!seq_lens || !params || b_max < 1) return PSK_ERR_INVALID_ARG;
  if (do_score && (!q || !summaries || !block_table)) return PSK_ERR_INVALID_ARG;
  if (do_select && !selected) return PSK_ERR_INVALID_ARG;
  const psk_select_params &sp = *params;
  if (sp.sink_pages < 0 || sp.window_pages < 1) return PSK_ERR_INVALID_ARG;
  if (sp.per_query_head != 0 && sp.per_query_head != 1) return PSK_ERR_INVALID_ARG;
  if (sp.mode == PSK_BUDGET_PER_SEQUENCE) {
    if (!sp.budgets) return PSK_ERR_INVALID_ARG;
  } else if (sp.mode == PSK_BUDGET_PAGES || sp.mode == PSK_BUDGET_FRACTION) {
    if (sp.mode == PSK_BUDGET_PAGES && sp.budget_pages < 1) return PSK_ERR_INVALID_ARG;
    if (sp.mode == PSK_BUDGET_FRACTION && !(sp.budget_fraction > 0.0 && sp.budget_fraction <= 1.0))
      return PSK_ERR_INVALID_ARG;
    if (scalar_mode_budget(sp, L.max_pages) > b_max) return PSK_ERR_INVALID_ARG;  // monotone in P
  } else {
    return PSK_ERR_INVALID_ARG;
  }
  if (do_score && (!aligned16(q) || !aligned16(summaries))) return PSK_ERR_INVALID_ARG;
  rc = check_gqa_compute(layout);
  if (rc != PSK_OK) return rc;
  if (gauss_stats && (L.latent || sp.per_query_head ||
                      !gauss_supported(L.dtype, L.head_dim, L.num_q_heads / L.num_kv_heads)))
    return PSK_ERR_UNSUPPORTED;
  // the units' layout: the cache's own, or its per-query-head view
  psk_layout U = L;
  int kv_shift = 0;
  if (sp.per_query_head && !per_query_head_view(L, &U, &kv_shift)) return PSK_ERR_UNSUPPORTED;
  ScorePlan plan;
  if (!plan_score(U, b_max, &plan, kv_shift)) return PSK_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < plan.ws_bytes) return PSK_ERR_WORKSPACE;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  ScoreArgs a;
  a.q = q;
  a.summaries = summaries;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.budgets = sp.mode == PSK_BUDGET_PER_SEQUENCE ? sp.budgets : nullptr;
  a.selected = selected;
  a.scores_out = scores_out;
  a.ws = workspace;
  a.counters = reinterpret_cast<uint32_t *>(ws + plan.off_counters);
  a.keys = reinterpret_cast<uint32_t *>(ws + plan.off_keys);
  a.key_stride = (L.max_pages + 3) & ~3;
  a.cand_key = reinterpret_cast<uint32_t *>(ws + plan.off_key);
  a.cand_page = reinterpret_cast<int32_t *>(ws + plan.off_page);
  a.cand_count = reinterpret_cast<int32_t *>(ws + plan.off_count);
  a.B = L.batch;
  a.H_q = L.num_q_heads;
  a.H_kv = U.num_kv_heads;
  a.H_kv_cache = L.num_kv_heads;
  a.kv_shift = kv_shift;
  a.D = L.head_dim;
  a.ps = L.page_size;
  a.nb = L.num_blocks;
  a.max_pages = L.max_pages;
  a.b_max = b_max;
  a.pchunk = plan.pchunk;
  a.stage_pages = plan.stage_pages;
  a.chunk = plan.chunk;
  a.n_chunks_max = plan.n_chunks_max;
  a.k_cap = plan.k_cap;
  a.scale = scale;
  a.sink = sp.sink_pages;
  a.window = sp.window_pages;
  a.budget_mode = sp.mode;
  a.budget_pages = sp.budget_pages;
  a.budget_frac = sp.budget_fraction;
  a.unit_budgets = nullptr;
  if (gauss_stats)
    return cuda_status(launch_gauss_score_select(a, gauss_stats, gauss_z, L.dtype, static_cast<cudaStream_t>(stream)));
  if (L.latent)
    return cuda_status(launch_mla_score_select(a, reinterpret_cast<uint16_t *>(ws + plan.off_qsplit),
                                               static_cast<cudaStream_t>(stream), stages));
  return cuda_status(launch_score_select(a, L.dtype, static_cast<cudaStream_t>(stream), stages));
}

int psk_page_score_select_ex(const psk_layout *layout, const void *q, const void *summaries,
                             const int32_t *block_table, const int32_t *seq_lens, const psk_select_params *params,
                             int32_t b_max, float scale, int32_t *selected, float *scores_out, void *workspace,
                             size_t workspace_bytes, psk_stream_t stream) {
  return score_select_common(layout, q, summaries, block_table, seq_lens, params, b_max, scale, selected, scores_out,
                             workspace, workspace_bytes, stream, kStageScore | kStageSelect);
}

int psk_page_score_select_gaussian(const psk_layout *layout, const void *q, const float *stats,
                                   const int32_t *block_table, const int32_t *seq_lens,
                                   const psk_select_params *params, int32_t b_max, float scale, float z,
                                   int32_t *selected, float *scores_out, void *workspace, size_t workspace_bytes,
                                   psk_stream_t stream) {
  if (!stats || !(z == z)) return PSK_ERR_INVALID_ARG;
  return score_select_common(layout, q, stats, block_table, seq_lens, params, b_max, scale, selected, scores_out,
                             workspace, workspace_bytes, stream, kStageScore | kStageSelect, stats, z);
}

int psk_page_score(const psk_layout *layout, const void *q, const void *summaries, const int32_t *block_table,
                   const int32_t *seq_lens, const psk_select_params *params, int32_t b_max, float scale,
                   float *scores_out, void *workspace, size_t workspace_bytes, psk_stream_t stream) {
  return score_select_common(layout, q, summaries, block_table, seq_lens, params, b_max, scale, nullptr, scores_out,
                             workspace, workspace_bytes, stream, kStageScore);
}

int psk_page_select(const psk_layout *layout, const int32_t *seq_lens, const psk_select_params *params,
                    int32_t b_max, int32_t *selected, void *workspace, size_t workspace_bytes, psk_stream_t stream) {
  return score_select_common(layout, nullptr, nullptr, nullptr, seq_lens, params, b_max, 0.f, selected, nullptr,
                             workspace, workspace_bytes, stream, kStageSelect);
}

// Workspace of the coverage selection: the score / select regions of the layout, then the
// per-page (max, sum) pairs, the fixed-point masses and the per-unit budgets.
struct CoveragePlan {
  ScorePlan sel;
  size_t off_pm, off_qmass, off_budgets, ws_bytes;
};
static bool plan_coverage(const psk_layout &L, int b_max, CoveragePlan *cp) {
  if (L.latent) return false;
  const int G = L.num_q_heads / L.num_kv_heads;
  if (!coverage_supported(L.dtype, L.head_dim, G)) return false;
  if (!plan_score(L, b_max, &cp->sel)) return false;
  const size_t units = (size_t)L.batch * L.num_kv_heads;
  size_t off = align_up(cp->sel.ws_bytes, 256);
  cp->off_pm = off;
  off = align_up(off + units * (size_t)L.max_pages * G * 2 * 4, 256);
  cp->off_qmass = off;
  off = align_up(off + units * (size_t)L.max_pages * 8, 256);
  cp->off_budgets = off;
  off = align_up(off + units * 4, 256);
  cp->ws_bytes = off;
  return true;
}

size_t psk_coverage_workspace_size(const psk_layout *layout, int32_t b_max) {
  if (check_layout(layout) != PSK_OK || check_gqa_compute(layout) != PSK_OK || b_max < 1) return 0;
  CoveragePlan cp;
  return plan_coverage(*layout, b_max, &cp) ? cp.ws_bytes : 0;
}

int psk_page_select_coverage(const psk_layout *layout, const void *q, const void *k_cache, const int32_t *block_table,
                             const int32_t *seq_lens, double coverage, int32_t sink_pages, int32_t window_pages,
                             int32_t b_max, float scale, int32_t *selected, float *masses_out, void *workspace,
                             size_t workspace_bytes, psk_stream_t stream) {
  int rc = check_layout(layout);
  if (rc != PSK_OK) return rc;
  const psk_layout &L = *layout;
  if (!q || !k_cache || !block_table || !seq_lens || !selected || b_max < 1) return PSK_ERR_INVALID_ARG;
  if (!(coverage > 0.0 && coverage <= 1.0) || sink_pages < 0 || window_pages < 1) return PSK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache)) return PSK_ERR_INVALID_ARG;
  rc = check_gqa_compute(layout);
  if (rc != PSK_OK) return rc;
  CoveragePlan cp;
  if (!plan_coverage(L, b_max, &cp)) return PSK_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < cp.ws_bytes) return PSK_ERR_WORKSPACE;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  ScoreArgs a = {};
  a.seq_lens = seq_lens;
  a.selected = selected;
  a.ws = workspace;
  a.counters = reinterpret_cast<uint32_t *>(ws + cp.sel.off_counters);
  a.keys = reinterpret_cast<uint32_t *>(ws + cp.sel.off_keys);
  a.key_stride = (L.max_pages + 3) & ~3;
  a.cand_key = reinterpret_cast<uint32_t *>(ws + cp.sel.off_key);
  a.cand_page = reinterpret_cast<int32_t *>(ws + cp.sel.off_page);
  a.cand_count = reinterpret_cast<int32_t *>(ws + cp.sel.off_count);
  a.B = L.batch;
  a.H_q = L.num_q_heads;
  a.H_kv = L.num_kv_heads;
  a.H_kv_cache = L.num_kv_heads;
  a.D = L.head_dim;
  a.ps = L.page_size;
  a.nb = L.num_blocks;
  a.max_pages = L.max_pages;
  a.b_max = b_max;
  a.chunk = cp.sel.chunk;
  a.n_chunks_max = cp.sel.n_chunks_max;
  a.k_cap = cp.sel.k_cap;
  a.sink = sink_pages;
  a.window = window_pages;
  a.budget_mode = PSK_BUDGET_PER_SEQUENCE;
  a.unit_budgets = reinterpret_cast<int32_t *>(ws + cp.off_budgets);
  CoverageArgs c = {};
  c.q = q;
  c.k_cache = k_cache;
  c.block_table = block_table;
  c.seq_lens = seq_lens;
  c.ws = workspace;
  c.pm = reinterpret_cast<float *>(ws + cp.off_pm);
  c.keys = a.keys;
  c.qmass = reinterpret_cast<unsigned long long *>(ws + cp.off_qmass);
  c.unit_budgets = reinterpret_cast<int32_t *>(ws + cp.off_budgets);
  c.masses_out = masses_out;
  c.B = L.batch;
  c.H_q = L.num_q_heads;
  c.H_kv = L.num_kv_heads;
  c.D = L.head_dim;
  c.ps = L.page_size;
  c.nb = L.num_blocks;
  c.max_pages = L.max_pages;
  c.b_max = b_max;
  c.key_stride = a.key_stride;
  c.sink = sink_pages;
  c.window = window_pages;
  c.scale = scale;
  c.coverage = coverage;
  return cuda_status(launch_coverage_select(c, a, L.dtype, static_cast<cudaStream_t>(stream)));
}

static int decode_common(const psk_layout *layout, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_table, const int32_t *seq_lens, const int32_t *selected,
                         int32_t b_max, float scale, void *out, void *workspace, size_t workspace_bytes,
                         psk_stream_t stream, bool per_query_head = false, bool v_host = false,
                         const void *v_hot = nullptr, const int32_t *v_slot = nullptr, int32_t n_slots = 0) {
  int rc = check_layout(layout);
  if (rc != PSK_OK) return rc;
  const psk_layout &L = *layout;
  if (!q || !k_cache || !block_table || !seq_lens || !out) return PSK_ERR_INVALID_ARG;
  if (L.latent ? v_cache != nullptr : v_cache == nullptr) return PSK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PSK_ERR_INVALID_ARG;
  rc = check_gqa_compute(layout);
  if (rc != PSK_OK) return rc;
  const bool dense = selected == nullptr;
  psk_layout U = L;  // the units' layout (per-query-head view for per-query-head rows)
  int kv_shift = 0;
  if (per_query_head && (dense || !per_query_head_view(L, &U, &kv_shift))) return PSK_ERR_UNSUPPORTED;
  // the value tier in host memory: sparse GQA decode, bf16, head_dim 128
  if (v_host && (dense || L.latent || L.dtype != PSK_BF16 || L.head_dim != 128)) return PSK_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (!plan_any_decode(U, dense ? L.max_pages : b_max, dense, &plan)) return PSK_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < plan.ws_bytes) return PSK_ERR_WORKSPACE;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  DecodeArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.selected = selected;
  a.out = out;
  a.ws = workspace;
  a.part_o = reinterpret_cast<float *>(ws + plan.off_o);
  a.part_ml = reinterpret_cast<float *>(ws + plan.off_ml);
  a.tickets = reinterpret_cast<uint32_t *>(ws + plan.off_tickets);
  a.B = L.batch;
  a.H_q = L.num_q_heads;
  a.H_kv = U.num_kv_heads;
  a.H_kv_cache = L.num_kv_heads;
  a.kv_shift = kv_shift;
  a.v_host = v_host ? 1 : 0;
  a.v_hot = v_hot;
  a.v_slot = v_slot;
  a.n_slots = n_slots;
  a.D = L.head_dim;
  a.D_v = L.v_head_dim;
  a.ps = L.page_size;
  a.nb = L.num_blocks;
  a.max_pages = L.max_pages;
  a.b_max = dense ? L.max_pages : b_max;
  a.sw = plan.sw;
  a.n_items_max = plan.n_items_max;
  a.flat = plan.flat;
  a.taper = plan.taper;
  a.counts = reinterpret_cast<int32_t *>(ws + plan.off_counts);
  a.scale = scale;
  if (L.latent) return cuda_status(launch_mla_decode(a, static_cast<cudaStream_t>(stream)));
  return cuda_status(launch_decode(a, L.dtype, static_cast<cudaStream_t>(stream)));
}

int psk_sparse_paged_decode(const psk_layout *layout, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_table, const int32_t *seq_lens, const int32_t *selected,
                            int32_t b_max, float scale, void *out, void *workspace, size_t workspace_bytes,
                            psk_stream_t stream) {
  if (!selected || b_max < 1) return PSK_ERR_INVALID_ARG;
  return decode_common(layout, q, k_cache, v_cache, block_table, seq_lens, selected, b_max, scale, out, workspace,
                       workspace_bytes, stream);
}

int psk_sparse_paged_decode_ex(const psk_layout *layout, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_table, const int32_t *seq_lens, const int32_t *selected,
                               int32_t b_max, float scale, uint32_t flags, void *out, void *workspace,
                               size_t workspace_bytes, psk_stream_t stream) {
  if (!selected || b_max < 1 || (flags & ~(PSK_DECODE_PER_QUERY_HEAD | PSK_DECODE_V_HOST)) != 0)
    return PSK_ERR_INVALID_ARG;
  return decode_common(layout, q, k_cache, v_cache, block_table, seq_lens, selected, b_max, scale, out, workspace,
                       workspace_bytes, stream, (flags & PSK_DECODE_PER_QUERY_HEAD) != 0,
                       (flags & PSK_DECODE_V_HOST) != 0);
}

int psk_sparse_paged_decode_tiered(const psk_layout *layout, const void *q, const void *k_cache,
                                   const void *v_cache_host, const void *v_hot, int32_t n_slots,
                                   const int32_t *v_slot, const int32_t *block_table, const int32_t *seq_lens,
                                   const int32_t *selected, int32_t b_max, float scale, void *out,
                                   void *workspace, size_t workspace_bytes, psk_stream_t stream) {
  if (!selected || b_max < 1 || !v_hot || !v_slot || n_slots < 1 || !aligned16(v_hot)) return PSK_ERR_INVALID_ARG;
  return decode_common(layout, q, k_cache, v_cache_host, block_table, seq_lens, selected, b_max, scale, out, workspace,
                       workspace_bytes, stream, false, true, v_hot, v_slot, n_slots);
}

int psk_value_tier_fill(const psk_layout *layout, const void *v_cache_host, const int32_t *block_table,
                        const int32_t *entries, int32_t n_entries, void *v_hot, int32_t n_slots, int32_t *v_slot,
                        void *workspace, size_t workspace_bytes, psk_stream_t stream) {
  int rc = check_layout(layout);
  if (rc != PSK_OK) return rc;
  const psk_layout &L = *layout;
  if (L.latent || L.dtype != PSK_BF16 || L.v_head_dim != 128) return PSK_ERR_UNSUPPORTED;
  if (n_entries < 0 || n_slots < 1 || !v_cache_host || !block_table || !v_hot || !v_slot || (n_entries > 0 && !entries))
    return PSK_ERR_INVALID_ARG;
  if (!aligned16(v_cache_host) || !aligned16(v_hot)) return PSK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWsHeader) return PSK_ERR_WORKSPACE;
  return cuda_status(launch_value_tier_fill(L, v_cache_host, block_table, entries, n_entries, v_hot, n_slots, v_slot,
                                            workspace, static_cast<cudaStream_t>(stream)));
}

int psk_dense_paged_decode(const psk_layout *layout, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens, float scale, void *out,
                           void *workspace, size_t workspace_bytes, psk_stream_t stream) {
  return decode_common(layout, q, k_cache, v_cache, block_table, seq_lens, nullptr, 0, scale, out, workspace,
                       workspace_bytes, stream);
}

}  // extern "C"
