// Selection pieces shared by the selection kernel (select.cu) and the coverage selection
// (coverage.cu): the unit budget and the layout of a selected row.
//
// Selection rule (LOCKS PKG-INFO, "How it works", Selection, and "Configuration (LocksConfig)";
// EntmaxKV README, "Two selection strategies", Top-k): the always-kept pages (first `sink`, last
// `window`) plus the k = b - |always kept| highest-scoring other pages, ties to the lower page
// index. The score kernels leave one 32-bit order key per (unit, page): larger score -> larger
// key, 0 for an always-kept page or a flagged bad block (never a candidate).
#pragma once

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {

// Budget of a sequence of P pages (at least the always-kept count in the scalar modes);
// budget_in: the sequence's entry of a.budgets in the per-sequence mode.
__device__ __forceinline__ int unit_budget(const ScoreArgs &a, int budget_in, int P, int n_forced) {
  if (a.budget_mode == PSK_BUDGET_FRACTION) {
    const int r = (int)ceil((double)P * a.budget_frac);  // IEEE double product, then the ceiling
    return max(n_forced, min(P, max(1, r)));
  }
  if (a.budget_mode == PSK_BUDGET_PAGES) return max(n_forced, min(P, a.budget_pages));
  return budget_in;
}

// Row of a unit with count < P selected pages: the first S pages, the `wrote` winners (written
// by the caller at sel_row + S, all inside [S, P - W)), the last W pages straight after them,
// then -1 to b_max. count < P implies S + W < P, so the two always-kept runs do not overlap.
// wrote < count - S - W happens only after a flagged bad block: the row is then shorter, and the
// -1 padding still comes only at its end (the decode reads a row up to its first -1). Threads
// t0, t0 + nt, ... of the caller's group write.
__device__ __forceinline__ void write_row_ends(int32_t *sel_row, int P, int wrote, int b_max, int S, int W, int t0,
                                               int nt) {
  for (int x = t0; x < S; x += nt) sel_row[x] = x;
  const int w0 = S + wrote;
  for (int x = t0; x < W; x += nt) sel_row[w0 + x] = P - W + x;
  for (int x = w0 + W + t0; x < b_max; x += nt) sel_row[x] = -1;
}

}  // namespace psk
