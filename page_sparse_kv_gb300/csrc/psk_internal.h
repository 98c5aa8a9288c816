// Launchers shared between the kernel translation units and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/psk.h"

namespace psk {

struct AppendArgs {
  const void *k_new;
  const void *v_new;
  const int32_t *start_pos;
  const int32_t *cu_new;
  void *k_cache;
  void *v_cache;
  void *summaries;    // k_min / k_max summaries (storage dtype), or NULL
  float *stats;       // fp32 [num_blocks, H_kv, 2, D] key mean / std per page, or NULL
  const int32_t *block_table;
  void *ws;
  int B, H_kv, D, D_v, ps, nb, max_pages;
};
cudaError_t launch_append(const AppendArgs &a, int dtype, int max_new, cudaStream_t s);

struct ScoreArgs {
  const void *q;
  const void *summaries;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *budgets;
  int32_t *selected;
  float *scores_out;
  void *ws;
  // workspace regions
  uint32_t *counters;     // [B * H_kv]
  uint32_t *keys;         // [B * H_kv, max_pages] selection keys written by the score kernel
  uint32_t *cand_key;     // [B * H_kv, n_chunks_max, k_cap]
  int32_t *cand_page;     // same shape
  int32_t *cand_count;    // [B * H_kv, n_chunks_max]
  int B, H_q, H_kv, D, ps, nb, max_pages, b_max;
  int key_stride;         // keys per (sequence, KV head) row of `keys`: max_pages rounded up to 4
  int pchunk;             // pages per streaming score CTA (body region)
  int body_chunks;        // score CTAs per (sequence, head group) in the body region (set at launch)
  int tail_pages;         // last pages of each sequence scored by the tail region (set at launch)
  int tail_chunk;         // pages per tail-region CTA (set at launch)
  int tail_chunks;        // tail-region CTAs per (sequence, head group) (set at launch)
  int stage_pages;        // pages per shared-memory stage of the score kernel
  int chunk;              // pages per selection CTA
  int n_chunks_max;
  int k_cap;              // candidates kept per chunk = min(max(1, b_max - 1), chunk): with sink_pages = 0
                          // only the tail page is always kept
  float scale;
  int sink, window;       // always-kept first (>= 0) / last (>= 1) pages
  int H_kv_cache;         // KV heads of the cache (H_kv above counts the units' heads)
  int kv_shift;           // unit head h reads cache head h >> kv_shift (log2 G when selecting per query head)
  int budget_mode;        // enum psk_budget_mode
  int budget_pages;       // PSK_BUDGET_PAGES
  double budget_frac;     // PSK_BUDGET_FRACTION
  const int32_t *unit_budgets;  // non-null: per-unit budgets (coverage mode) instead of budgets[i]
  int mma_hpc;            // unit heads per CTA of the tensor-core score kernel (set at launch)
};

// Page p of a sequence of P pages is always kept: one of the first `sink` or the last `window`.
__host__ __device__ inline bool always_kept(int p, int P, int sink, int window) {
  return p < sink || p >= P - window;
}
struct ScorePlan {
  int pchunk, stage_pages, chunk, n_chunks_max, k_cap;
  size_t ws_bytes;
  size_t off_counters, off_keys, off_key, off_page, off_count, off_qsplit;
};
// kv_shift > 0: L is the per-query-head view (num_kv_heads = num_q_heads), whose unit heads share
// cache heads 2^kv_shift at a time.
bool plan_score(const psk_layout &L, int b_max, ScorePlan *plan, int kv_shift = 0);
// Stages of a score / select launch: the page-score kernels (keys into the workspace, scores_out)
// and the selection kernel (keys -> selected rows).
constexpr int kStageScore = 1, kStageSelect = 2;
constexpr int kMergeCap = 8192;  // candidates the selection's merge CTA holds (shared memory)
cudaError_t launch_page_select(const ScoreArgs &a, cudaStream_t s, bool first_of_call = false);
cudaError_t launch_score_select(const ScoreArgs &a, int dtype, cudaStream_t s, int stages = kStageScore | kStageSelect);
bool score_supported(int dtype, int D, int G);

struct DecodeArgs {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *selected;  // NULL: dense (every page)
  void *out;
  void *ws;
  float *part_o;       // [B * H_kv, n_items_max, G, D_v] per-item partial O (unnormalised)
  float *part_ml;      // [B * H_kv, n_items_max, G, 2] per-item (m, l)
  uint32_t *tickets;   // [B * H_kv] merge tickets (zero between calls)
  int B, H_q, H_kv, D, D_v, ps, nb, max_pages;
  int b_max;           // entries per selected row (sparse)
  int H_kv_cache;      // KV heads of the cache (H_kv above counts the units' heads)
  int kv_shift;        // unit head h reads cache head h >> kv_shift
  int v_host;          // 1: v_cache is host memory read over NVLink-C2C (sparse split, bf16, D = 128)
  const void *v_hot;   // v_host: resident HBM copies of full pages' V rows [n_slots, ps, D_v], or NULL
  const int32_t *v_slot;  // v_host: slot of (sequence, cache head, logical page) [B, H_kv_cache, max_pages], -1 = host
  int n_slots;
  int sw;              // list entries per item (split layout)
  int n_items_max;     // items per unit (split layout)
  int32_t *counts;     // [B * H_kv] list entries per unit (flat layout, sparse)
  int flat;            // 1: flat layout (the units' lists cut into equal shares of a persistent grid)
  int taper;           // split layout: 1 = split lengths halve every two splits (see split_len)
  float scale;
};
struct DecodePlan {
  int sw, n_items_max, flat, taper;
  size_t ws_bytes, off_o, off_ml, off_tickets, off_counts;
};
bool plan_decode(const psk_layout &L, int entries, bool dense, DecodePlan *plan);
// Split layout: list entries of split s, and where it starts. With taper, the lengths are
// sw, sw, sw/2, sw/2, sw/4, ... (never below min(8, sw)): CTAs launch split-major, so the last
// CTAs of the grid carry the shortest pieces.
__host__ __device__ inline int split_len(int s, int sw, int taper) {
  if (!taper) return sw;
  const int floor_len = sw < 8 ? sw : 8;
  const int v = (s >> 1) >= 31 ? 0 : (sw >> (s >> 1));
  return v > floor_len ? v : floor_len;
}
__host__ __device__ inline int split_off(int s, int sw, int taper) {
  if (!taper) return s * sw;
  int o = 0;
  for (int j = 0; j < s; ++j) o += split_len(j, sw, 1);
  return o;
}
cudaError_t launch_decode(const DecodeArgs &a, int dtype, cudaStream_t s);
// Copies listed (sequence, cache head, page) V rows of a host value cache into hot-buffer slots
// and records the slots (slot < 0: the entry is evicted); see psk_value_tier_fill.
cudaError_t launch_value_tier_fill(const psk_layout &L, const void *v_host, const int32_t *block_table,
                                   const int32_t *entries, int n_entries, void *v_hot, int n_slots, int32_t *v_slot,
                                   void *ws, cudaStream_t s);
bool decode_supported(int dtype, int D, int D_v, int G, int ps);

// Gaussian page score from the mean / std summaries (gauss.cu): keys for the selection kernel
cudaError_t launch_gauss_score_select(const ScoreArgs &a, const float *stats, float z, int dtype, cudaStream_t s);
bool gauss_supported(int dtype, int D, int G);

// adaptive per-head coverage over exact page masses (coverage.cu)
struct CoverageArgs {
  const void *q;
  const void *k_cache;
  const int32_t *block_table;
  const int32_t *seq_lens;
  void *ws;
  float *pm;                   // [B * H_kv, max_pages, G, 2] per-page (max, sum of 2^(x - max)) per query head
  uint32_t *keys;              // the selection keys (ScoreArgs::keys)
  unsigned long long *qmass;   // [B * H_kv, max_pages] page masses in 2^-40 units
  int32_t *unit_budgets;       // [B * H_kv] budget of each unit for the selection
  float *masses_out;           // optional [B * H_kv, max_pages] page masses
  int B, H_q, H_kv, D, ps, nb, max_pages, b_max, key_stride, sink, window;
  float scale;
  double coverage;
};
bool coverage_supported(int dtype, int D, int G);
cudaError_t launch_coverage_select(const CoverageArgs &c, const ScoreArgs &sel, int dtype, cudaStream_t s);

// latent (MLA) form on the tensor cores
bool mla_supported(const psk_layout &L);
size_t mla_qsplit_bytes(const psk_layout &L);
cudaError_t launch_mla_score_select(const ScoreArgs &a, uint16_t *qsplit, cudaStream_t s,
                                    int stages = kStageScore | kStageSelect);
bool plan_mla_decode(const psk_layout &L, int entries, DecodePlan *plan);
cudaError_t launch_mla_decode(const DecodeArgs &a, cudaStream_t s);

}  // namespace psk
