// Selection pieces shared by the selection kernel (select.cu) and the score kernel's fused
// selection (score_select.cu): the unit budget, the layout of a selected row, and a one-warp
// top-k over a unit's keys.
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

constexpr int kSelBatch = 8;  // four-key groups each lane loads at once in warp_select_unit's passes

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

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// One warp selects unit `unit` of sequence i (P pages, 1 <= P <= a.key_stride) from its keys
// a.keys[unit * key_stride + p], p < P, and writes the unit's selected row exactly as the
// selection kernel does. hist: 256 ints of shared memory owned by this warp. Keys are read with
// L2-only loads (other CTAs wrote them). Radix select: MSB-first 8-bit digits from the highest
// bit where the smallest and largest candidate keys differ; the digit whose bin crosses the
// number of keys still needed is fixed, and the select stops once that bin holds exactly the keys
// still needed. Then the winners ("key > T, plus the first need_eq keys equal to T") are written
// in ascending page order. Every pass issues kSelBatch independent loads per lane before using
// them, so a pass over P keys costs about P / (128 kSelBatch) L2 round trips.
__device__ __forceinline__ void warp_select_unit(const ScoreArgs &a, int unit, int P, int budget_in, int *hist) {
  const int lane = threadIdx.x & 31;
  int32_t *sel_row = a.selected + (size_t)unit * a.b_max;
  const int n_forced = min(P, a.sink + a.window);
  const int budget = unit_budget(a, budget_in, P, n_forced);
  if (budget < n_forced || budget > a.b_max) {
    if (lane == 0) set_status(a.ws, PSK_DEV_BAD_BUDGET);
    for (int x = lane; x < a.b_max; x += 32) sel_row[x] = -1;
    return;
  }
  const int count = min(budget, P);
  if (count >= P) {  // every page is kept
    for (int x = lane; x < a.b_max; x += 32) sel_row[x] = x < P ? x : -1;
    return;
  }
  const int k_free = count - n_forced;  // count < P implies n_forced = sink + window < P
  const uint32_t *krow = a.keys + (size_t)unit * a.key_stride;  // 16-byte aligned (key_stride: x4)
  const int n4 = (P + 3) >> 2;
  // keys of the four-key group g (zero past P)
  auto load4 = [&](int g) -> uint4 {
    uint4 k = __ldcg(reinterpret_cast<const uint4 *>(krow) + g);
    const int p = g * 4;
    if (p + 3 >= P) {
      if (p + 0 >= P) k.x = 0u;
      if (p + 1 >= P) k.y = 0u;
      if (p + 2 >= P) k.z = 0u;
      if (p + 3 >= P) k.w = 0u;
    }
    return k;
  };
  int wrote = 0;
  if (k_free > 0) {
    // count, min and max of the candidate keys
    uint32_t cnt = 0, lo = 0xFFFFFFFFu, hi = 0u;
    for (int g0 = lane; g0 < n4; g0 += 32 * kSelBatch) {
      uint4 kb[kSelBatch];
#pragma unroll
      for (int b = 0; b < kSelBatch; ++b) kb[b] = g0 + 32 * b < n4 ? load4(g0 + 32 * b) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int b = 0; b < kSelBatch; ++b) {
        const uint32_t ks[4] = {kb[b].x, kb[b].y, kb[b].z, kb[b].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (ks[j] != 0u) {
            ++cnt;
            lo = min(lo, ks[j]);
            hi = max(hi, ks[j]);
          }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const bool take_all = (int)cnt <= k_free;
    uint32_t T = 0u;
    int need = k_free;
    if (!take_all) {
      const uint32_t diff = lo ^ hi;
      const int top = diff ? 31 - __clz(diff) : 0;
      int shift = top >= 7 ? top - 7 : 0;
      uint32_t prefix = shift + 8 >= 32 ? 0u : (lo >> (shift + 8)) << (shift + 8);
      uint32_t mask = shift + 8 >= 32 ? 0u : (0xFFFFFFFFu << (shift + 8));
#pragma unroll 1
      for (;;) {
#pragma unroll
        for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0;
        __syncwarp();
        for (int g0 = lane; g0 < n4; g0 += 32 * kSelBatch) {
          uint4 kb[kSelBatch];
#pragma unroll
          for (int b = 0; b < kSelBatch; ++b)
            kb[b] = g0 + 32 * b < n4 ? load4(g0 + 32 * b) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int b = 0; b < kSelBatch; ++b) {
            const uint32_t ks[4] = {kb[b].x, kb[b].y, kb[b].z, kb[b].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (ks[j] != 0u && (ks[j] & mask) == prefix) atomicAdd(&hist[(ks[j] >> shift) & 255u], 1);
          }
        }
        __syncwarp();
        // lane l owns the digits 255 - 8l .. 248 - 8l: descending digit order is lane order
        int c[8], s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - lane * 8 - j];
          s += c[j];
        }
        const int incl = warp_incl_scan(s, lane);
        const int excl = incl - s;
        const unsigned hit = __ballot_sync(0xffffffffu, excl < need && incl >= need);
        const int src = __ffs(hit) - 1;
        int d = 0, above = 0, in_bin = 0;
        if (lane == src) {
          int run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (in_bin == 0 && run + c[j] >= need && c[j] > 0) {
              d = 255 - lane * 8 - j;
              above = run;
              in_bin = c[j];
            }
            run += c[j];
          }
        }
        d = __shfl_sync(0xffffffffu, d, src);
        above = __shfl_sync(0xffffffffu, above, src);
        in_bin = __shfl_sync(0xffffffffu, in_bin, src);
        need -= above;
        prefix |= static_cast<uint32_t>(d) << shift;
        mask |= 255u << shift;
        __syncwarp();  // every lane has read hist before the next pass clears it
        if (shift == 0) break;
        if (in_bin == need) {
          // every key of the chosen bin is taken, and so is every key above it: the selection is
          // "key >= prefix" (prefix has zeros below this digit), with no tie left to break
          prefix = prefix == 0u ? 0u : prefix - 1u;
          need = 0;
          break;
        }
        shift = shift >= 8 ? shift - 8 : 0;  // an overlap with bits already fixed is harmless
      }
      T = prefix;
    }
    // winners in ascending page order: lane l holds pages 4l .. 4l + 3 of each 128-page block
    int run_eq = 0;
    int32_t *dst = sel_row + a.sink;
    uint4 next = lane < n4 ? load4(lane) : make_uint4(0u, 0u, 0u, 0u);
    for (int g0 = 0; g0 < n4; g0 += 32) {
      const int g = g0 + lane;
      const uint4 k = next;  // this block's keys; the next block's load is in flight meanwhile
      next = g + 32 < n4 ? load4(g + 32) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t ks[4] = {k.x, k.y, k.z, k.w};
      int eq = 0;
      if (!take_all) {
#pragma unroll
        for (int j = 0; j < 4; ++j) eq += (ks[j] != 0u && ks[j] == T);
      }
      const int eq_incl = warp_incl_scan(eq, lane);
      int eq_rank = run_eq + eq_incl - eq;
      bool take[4];
      int nt = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (take_all) {
          take[j] = ks[j] != 0u;
        } else {
          take[j] = ks[j] > T;
          if (ks[j] != 0u && ks[j] == T) take[j] = eq_rank++ < need;
        }
        nt += take[j];
      }
      const int t_incl = warp_incl_scan(nt, lane);
      int w = wrote + t_incl - nt;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (take[j]) dst[w++] = g * 4 + j;
      run_eq += __shfl_sync(0xffffffffu, eq_incl, 31);
      wrote += __shfl_sync(0xffffffffu, t_incl, 31);
    }
  }
  __syncwarp();
  write_row_ends(sel_row, P, wrote, a.b_max, a.sink, a.window, lane, 32);
}

}  // namespace psk
