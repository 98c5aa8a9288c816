// Stage 3: top-b page selection from the score kernel's keys (GQA and latent caches).
//
// Selection (LOCKS PKG-INFO, "How it works", Selection: a static top-b per (layer, KV head);
// sink and recent pages always kept and counted inside b; "Configuration (LocksConfig)":
// sink_pages / window_pages and the budget modes; EntmaxKV README, "Two selection strategies",
// Top-k: the budget includes the always-attended tail page, pages kept per query head; ties to
// the lower logical page index).
//
// The score kernel leaves one 32-bit order key per (unit, page) in the workspace: the fp32
// score's bits made unsigned-orderable, 0 for an always-kept page or a flagged bad block. A
// unit's free pages are the top k = b - |always kept| nonzero keys, ties to the lower index.
//
// page_select_kernel: one CTA of kSelThreads (384) per (unit head, chunk of up to a.chunk
// pages, sequence), four per SM, so all the CTAs of a large batch are resident at once. The
// CTA copies the chunk's keys (L2-resident after the score kernel) to shared memory with their
// count, min and max, then finds the k-th largest by an MSB-first radix select with 8-bit
// digits starting at the highest bit where min and max differ: the warps count into
// kHistCopies shared histograms, and warps 0..7 own one digit each (digit 255 - thread) to sum
// and clear the copies and scan the digits in descending order. The select stops as soon as
// the chosen digit's bin holds exactly the keys still needed. Ties at the threshold go to the
// lowest indices through a block scan in index order, and the winners are written in
// ascending page order. A unit larger than one chunk writes each chunk's winners; the last CTA
// of the unit to finish (an atomic ticket, no waiting) merges them with a second radix select:
// the top k of the union of the chunks' top k is the top k, since keys are unique once ties
// are ordered by page index.
// A globaltimer trace of every CTA on the batched workload (512 units, 2143 keys median): the
// key load with its statistics takes 2.7 us, the radix passes (two for most units) 6.3 us and
// the compaction 2.0 us, each stretched by the four CTAs sharing an SM; 256-thread CTAs
// (18.2 us for the kernel), 512 threads at three CTAs per SM and warp-aggregated histogram
// atomics (__match_any_sync, 22.2 us) measured slower than this form (16.8 us).
// The output row is: the first sink pages, the winners (ascending), the last window pages, -1.
#include <algorithm>

#include "psk_common.cuh"
#include "psk_internal.h"
#include "select_common.cuh"

namespace psk {
namespace {

constexpr int kSelThreads = 384;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kDigits = 256;      // 8-bit radix digits
constexpr int kHistCopies = 8;    // warp w counts into histogram copy w % kHistCopies
static_assert(kSelThreads >= kDigits && kSelWarps <= 32, "the digit phase uses the first 256 threads");

// Shared scratch of the block helpers.
struct SelScratch {
  int wsum[kSelWarps + 1];   // per-warp totals of a scan
  int dig[3 + kDigits / 32]; // chosen digit, keys above it, its bin's count; digit-phase warp totals
  uint32_t red[3 * kSelWarps];
  int flag_last;
};

// Exclusive prefix of x over the block in thread order, and the block total. Two barriers; the
// caller separates consecutive uses with a barrier of its own.
__device__ int block_excl_scan(int x, SelScratch &sc, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < kSelWarps ? sc.wsum[lane] : 0;
    int w = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSelWarps) sc.wsum[lane] = w - v;
    if (lane == 31) sc.wsum[kSelWarps] = w;
  }
  __syncthreads();
  if (total) *total = sc.wsum[kSelWarps];
  return sc.wsum[warp] + incl - x;
}

// Count, min and max of the nonzero keys the threads hold (c, lo, hi), over the block. Two
// barriers.
__device__ void block_stats(uint32_t c, uint32_t lo, uint32_t hi, SelScratch &sc, int *count, uint32_t *kmin,
                            uint32_t *kmax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    c += __shfl_xor_sync(0xffffffffu, c, o);
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sc.red[warp] = c;
    sc.red[kSelWarps + warp] = lo;
    sc.red[2 * kSelWarps + warp] = hi;
  }
  __syncthreads();
  c = 0;
  lo = 0xFFFFFFFFu;
  hi = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    c += sc.red[w];
    lo = min(lo, sc.red[kSelWarps + w]);
    hi = max(hi, sc.red[2 * kSelWarps + w]);
  }
  *count = (int)c;
  *kmin = lo;
  *kmax = hi;
  __syncthreads();  // red is reused by the next call
}

// Radix select over keys[0..n) in shared memory (key 0 = not a candidate): the k-th largest
// key T and how many keys equal to T belong to the top k (the lowest-indexed ones), returned
// as the rule "key > T, plus the first need_eq keys equal to T". Requires 1 <= k <= the number
// of nonzero keys, and kmin / kmax = the smallest / largest nonzero key. hist: kHistCopies x
// kDigits ints, zero on entry and on return. Three barriers per pass.
__device__ void radix_select(const uint32_t *keys, int n, int k, uint32_t kmin, uint32_t kmax, int *hist,
                             SelScratch &sc, uint32_t *T_out, int *need_eq_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t diff = kmin ^ kmax;
  const int top = diff ? 31 - __clz(diff) : 0;  // highest differing bit: the bits above are common
  int shift = top >= 7 ? top - 7 : 0;
  uint32_t prefix = shift + 8 >= 32 ? 0u : (kmin >> (shift + 8)) << (shift + 8);
  uint32_t mask = shift + 8 >= 32 ? 0u : (0xFFFFFFFFu << (shift + 8));
  int need = k;
  int *myhist = hist + (warp % kHistCopies) * kDigits;
#pragma unroll 1
  for (;;) {
    for (int x = tid; x < n; x += kSelThreads) {
      const uint32_t key = keys[x];
      if (key != 0u && (key & mask) == prefix) atomicAdd(&myhist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    // threads 0..255 own digits 255..0: descending digit order is thread order
    const int bin = kDigits - 1 - tid;
    int v = 0, incl = 0;
    if (tid < kDigits) {
#pragma unroll
      for (int c = 0; c < kHistCopies; ++c) {
        v += hist[c * kDigits + bin];
        hist[c * kDigits + bin] = 0;
      }
      incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) sc.dig[3 + warp] = incl;
    }
    __syncthreads();
    if (tid < kDigits) {
      for (int w = 0; w < warp; ++w) incl += sc.dig[3 + w];
      const int excl = incl - v;
      if (excl < need && incl >= need) {
        sc.dig[0] = bin;
        sc.dig[1] = excl;
        sc.dig[2] = v;
      }
    }
    __syncthreads();
    const int d = sc.dig[0];
    need -= sc.dig[1];
    const int in_bin = sc.dig[2];
    prefix |= static_cast<uint32_t>(d) << shift;
    mask |= 255u << shift;
    if (shift == 0) break;
    if (in_bin == need) {
      // every key of the chosen bin is taken, and so is every key above it: the selection is
      // "key >= prefix" (prefix has zeros below this digit), with no tie left to break
      prefix = prefix == 0u ? 0u : prefix - 1u;
      need = 0;
      break;
    }
    shift = shift >= 8 ? shift - 8 : 0;  // an overlap with bits already fixed is harmless
    __syncthreads();                     // dig is rewritten by the next pass
  }
  __syncthreads();  // every thread has read dig before it is reused
  *T_out = prefix;
  *need_eq_out = need;
}

// Writes, in index order, every key the rule takes (take_all: every nonzero key; otherwise
// key > T, or key == T among the first need_eq such keys) as a page id (pages ? pages[x] :
// page_base + x) to out_page, and the key to out_key when given. Returns the count. Each thread
// takes a contiguous run of indices; one block scan of the packed per-thread counts
// (equal << 16 | greater, both <= 16384) gives every thread its output position.
__device__ int compact_taken(const uint32_t *keys, const int32_t *pages, int page_base, int n, bool take_all,
                             uint32_t T, int need_eq, uint32_t *out_key, int32_t *out_page, SelScratch &sc) {
  const int tid = threadIdx.x;
  const int per = (n + kSelThreads - 1) / kSelThreads;
  const int x0 = min(n, tid * per), x1 = min(n, x0 + per);
  int gt = 0, eq = 0;
  for (int x = x0; x < x1; ++x) {
    const uint32_t key = keys[x];
    if (take_all) {
      gt += key != 0u;
    } else {
      gt += key > T;
      eq += key == T;
    }
  }
  int total;
  const int pre = block_excl_scan((eq << 16) | gt, sc, &total);
  int seen = pre >> 16;
  int w = (pre & 0xFFFF) + (take_all ? 0 : min(seen, need_eq));
  for (int x = x0; x < x1; ++x) {
    const uint32_t key = keys[x];
    bool take;
    if (take_all) {
      take = key != 0u;
    } else {
      take = key > T;
      if (key == T) take = (seen++ < need_eq);
    }
    if (take) {
      if (out_key) out_key[w] = key;
      out_page[w] = pages ? pages[x] : page_base + x;
      ++w;
    }
  }
  return (total & 0xFFFF) + (take_all ? 0 : min(total >> 16, need_eq));
}

__global__ void __launch_bounds__(kSelThreads, 4) page_select_kernel(ScoreArgs a) {
  pdl_wait();  // dependents are released when this grid completes
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ int hist[kHistCopies * kDigits];  // zero between radix selects
  __shared__ SelScratch sc;

  const int h = blockIdx.x, c = blockIdx.y, i = blockIdx.z;
  const int unit = i * a.H_kv + h;
  const int tid = threadIdx.x;
  const int seq_len = a.seq_lens[i];
  // the budget load is issued together with the length's (both are one L2 round trip)
  const int budget_in =
      a.budget_mode == PSK_BUDGET_PER_SEQUENCE ? (a.unit_budgets ? a.unit_budgets[unit] : a.budgets[i]) : 0;
  const int P = (seq_len + a.ps - 1) / a.ps;
  int32_t *sel_row = a.selected + (size_t)unit * a.b_max;

  if (seq_len < 1 || P > a.max_pages) {
    if (c == 0) {
      if (tid == 0) set_status(a.ws, PSK_DEV_BAD_SEQLEN);
      for (int x = tid; x < a.b_max; x += kSelThreads) sel_row[x] = -1;
    }
    return;
  }
  const int n_forced = min(P, a.sink + a.window);
  const int budget = unit_budget(a, budget_in, P, n_forced);
  if (budget < n_forced || budget > a.b_max) {
    if (c == 0) {
      if (tid == 0) set_status(a.ws, PSK_DEV_BAD_BUDGET);
      for (int x = tid; x < a.b_max; x += kSelThreads) sel_row[x] = -1;
    }
    return;
  }
  const int count = min(budget, P);
  if (count >= P) {  // every page is kept
    if (c == 0)
      for (int x = tid; x < a.b_max; x += kSelThreads) sel_row[x] = x < P ? x : -1;
    return;
  }
  const int nch = (P + a.chunk - 1) / a.chunk;
  if (c >= nch) return;
  const int k_free = count - n_forced;  // count < P implies n_forced = sink + window < P

  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw);
  const int p0 = c * a.chunk;
  const int n = min(P, p0 + a.chunk) - p0;
  const uint32_t *krow = a.keys + (size_t)unit * a.key_stride + p0;  // 16-byte aligned (stride, p0: x4)
  for (int x = tid; x < kHistCopies * kDigits; x += kSelThreads) hist[x] = 0;
  int total_valid;
  uint32_t kmin, kmax;
  {  // keys to shared memory, four per load, with the count, min and max of the nonzero ones
    uint32_t cnt = 0, lo = 0xFFFFFFFFu, hi = 0u;
    auto take = [&](uint32_t k) {
      if (k != 0u) {
        ++cnt;
        lo = min(lo, k);
        hi = max(hi, k);
      }
    };
    const int n4 = n >> 2;
    for (int x = tid; x < n4; x += kSelThreads) {
      const uint4 k4 = __ldcg(reinterpret_cast<const uint4 *>(krow) + x);
      reinterpret_cast<uint4 *>(keys)[x] = k4;
      take(k4.x);
      take(k4.y);
      take(k4.z);
      take(k4.w);
    }
    for (int x = 4 * n4 + tid; x < n; x += kSelThreads) {
      const uint32_t k = __ldcg(krow + x);
      keys[x] = k;
      take(k);
    }
    block_stats(cnt, lo, hi, sc, &total_valid, &kmin, &kmax);  // its barrier also publishes keys[] and hist
  }
  int wrote = 0;
  if (k_free > 0) {
    uint32_t thr = 0;
    int need_eq = 0;
    const bool take_all = total_valid <= k_free;
    if (!take_all) radix_select(keys, n, k_free, kmin, kmax, hist, sc, &thr, &need_eq);
    if (nch == 1) {
      wrote = compact_taken(keys, nullptr, p0, n, take_all, thr, need_eq, nullptr, sel_row + a.sink, sc);
      write_row_ends(sel_row, P, wrote, a.b_max, a.sink, a.window, tid, kSelThreads);
      return;
    }
    const int slot = unit * a.n_chunks_max + c;
    wrote = compact_taken(keys, nullptr, p0, n, take_all, thr, need_eq, a.cand_key + (size_t)slot * a.k_cap,
                          a.cand_page + (size_t)slot * a.k_cap, sc);
    if (tid == 0) a.cand_count[slot] = wrote;
  } else {
    if (nch == 1) {
      write_row_ends(sel_row, P, 0, a.b_max, a.sink, a.window, tid, kSelThreads);
      return;
    }
    if (tid == 0) a.cand_count[unit * a.n_chunks_max + c] = 0;
  }

  // ---- the last CTA of the unit merges ---------------------------------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.counters[unit], 1u);
    sc.flag_last = (prev == (unsigned)(nch - 1));
  }
  __syncthreads();
  if (!sc.flag_last) return;
  __threadfence();
  if (tid == 0) a.counters[unit] = 0u;

  uint32_t *mkey = reinterpret_cast<uint32_t *>(smem_raw);
  int32_t *mpage = reinterpret_cast<int32_t *>(smem_raw + sizeof(uint32_t) * kMergeCap);
  int *moff = reinterpret_cast<int *>(smem_raw + 2 * sizeof(uint32_t) * kMergeCap);  // [nch + 1]
  // every chunk's winner count at once, then their offsets (a walk over the chunks that waited
  // for each count before the next copy took 16 dependent round trips at 16 chunks)
  const int *cnt_row = a.cand_count + (size_t)unit * a.n_chunks_max;
  for (int cc = tid; cc < nch; cc += kSelThreads) moff[cc + 1] = __ldcg(cnt_row + cc);
  __syncthreads();
  if (tid == 0) {
    moff[0] = 0;
    for (int cc = 0; cc < nch; ++cc) moff[cc + 1] += moff[cc];
  }
  __syncthreads();
  const int n_c = moff[nch];
  const uint32_t *ck_row = a.cand_key + (size_t)unit * a.n_chunks_max * a.k_cap;
  const int32_t *cp_row = a.cand_page + (size_t)unit * a.n_chunks_max * a.k_cap;
  for (int idx = tid; idx < nch * a.k_cap; idx += kSelThreads) {
    const int cc = idx / a.k_cap, x = idx - cc * a.k_cap;
    if (x < moff[cc + 1] - moff[cc]) {
      mkey[moff[cc] + x] = __ldcg(ck_row + idx);
      mpage[moff[cc] + x] = __ldcg(cp_row + idx);
    }
  }
  __syncthreads();
  wrote = 0;
  if (k_free > 0) {
    uint32_t thr = 0;
    int need_eq = 0;
    const bool take_all = n_c <= k_free;
    if (!take_all) {
      uint32_t c2 = 0, lo = 0xFFFFFFFFu, hi = 0u;
      for (int x = tid; x < n_c; x += kSelThreads) {
        const uint32_t k = mkey[x];
        c2 += k != 0u;
        if (k != 0u) {
          lo = min(lo, k);
          hi = max(hi, k);
        }
      }
      int nz;
      uint32_t mlo, mhi;
      block_stats(c2, lo, hi, sc, &nz, &mlo, &mhi);
      radix_select(mkey, n_c, k_free, mlo, mhi, hist, sc, &thr, &need_eq);
    }
    wrote = compact_taken(mkey, mpage, 0, n_c, take_all, thr, need_eq, nullptr, sel_row + a.sink, sc);
  }
  write_row_ends(sel_row, P, wrote, a.b_max, a.sink, a.window, tid, kSelThreads);
}

}  // namespace

cudaError_t launch_page_select(const ScoreArgs &a, cudaStream_t s, bool first_of_call) {
  // keys of one chunk; the merge buffer only when a unit spans several chunks (the smaller
  // footprint keeps every CTA of a one-chunk call resident at once)
  const size_t keys_bytes = (size_t)std::min(a.chunk, a.max_pages) * 4;
  const size_t merge_bytes = (size_t)kMergeCap * 8 + (size_t)(a.n_chunks_max + 1) * 4;  // keys, pages, offsets
  const size_t smem = a.n_chunks_max == 1 ? keys_bytes : std::max<size_t>(keys_bytes, merge_bytes);
  dim3 grid(a.H_kv, a.n_chunks_max, a.B);
  return launch_kernel(first_of_call, page_select_kernel, grid, kSelThreads, smem, s, a);
}

}  // namespace psk
