// Stage 2: Quest-style page scores (GQA caches); stage 3, the selection, is in select.cu.
//
// Score (EntmaxKV README, "Two selection strategies", Top-k; kernels/page_criticality.py):
//   score[i,h,p] = scale * max_{g in group(h)} sum_d max(q_gd * kmin_pd, q_gd * kmax_pd)
// The kernels evaluate each term as max(q,0) * kmax + min(q,0) * kmin, which equals
// max(q * kmin, q * kmax) exactly whenever kmin <= kmax (one of the two products is +-0),
// so every kept product is the same fp32 product; accumulation is fp32.
//
// Two kernels stream the summaries, one CTA per (chunk of pages, sequence, group of up to 8 KV
// heads), so a page's summaries for all the group's heads (one 4 KB run at D = 128 bf16) are
// read together:
// - page_score_mma_kernel (bf16 caches, per-KV-head units; the default): the sum over a
//   summary row is one dot product of length 2D, taken on the tensor cores by warp-level
//   mma.sync over 16 (page, head) rows at a time (see its section below).
// - page_score_kernel (fp32 caches, the per-query-head view, and bf16 when PSK_SCORE_MMA=0):
//   warp w scores KV head w % 8 of the group; a (page, head) summary row is read by
//   LPP = D * sizeof(T) / 16 lanes with one 16-byte load each and summed with FMAs (bf16: mixed
//   fma.f32.bf16 on the raw bf16 pairs; fp32: packed fp32x2 FMAs). Partial sums are reduced
//   across the LPP lanes by a transposing butterfly (each step halves the values a lane
//   carries), then the group max is taken across the lanes that ended up holding different
//   query heads.
// Both write one 32-bit order key per page to the workspace (0 = an always-kept page, or a
// flagged bad block), which the selection kernel reads.
#include <algorithm>

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr int kThreads = 256;  // score kernel: eight warps, one KV head of the group each
constexpr int kWarps = kThreads / 32;

// ------------------------------------------------------------------------------------
// reductions across the LPP lanes of one page
// ------------------------------------------------------------------------------------
// v[g] holds this lane's partial sum for query head g. Returns, on every lane of the page
// group, max over g of the full sums.
template <int G, int LPP>
__device__ __forceinline__ float group_score(float (&v)[G], int lane) {
  int L = G;
#pragma unroll
  for (int mask = LPP / 2; mask >= 1; mask >>= 1) {
    if (L > 1) {
      const int half = L / 2;
      const bool upper = (lane & mask) != 0;
#pragma unroll
      for (int k = 0; k < (G > 1 ? G / 2 : 1); ++k) {
        if (k < half) {
          const float mine = upper ? v[k + half] : v[k];
          const float other = upper ? v[k] : v[k + half];
          v[k] = mine + __shfl_xor_sync(0xffffffffu, other, mask);
        }
      }
      L = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
    }
  }
  float mx = v[0];
#pragma unroll
  for (int k = 1; k < G; ++k)
    if (k < L) mx = fmaxf(mx, v[k]);
  // max over the lanes that carried different heads (the masks used by the transposing steps)
  constexpr int kLogG = (G >= 8) ? 3 : (G >= 4) ? 2 : (G >= 2) ? 1 : 0;
  constexpr int kLogL = (LPP >= 32) ? 5 : (LPP >= 16) ? 4 : (LPP >= 8) ? 3 : (LPP >= 4) ? 2 : (LPP >= 2) ? 1 : 0;
  constexpr int kSteps = kLogG < kLogL ? kLogG : kLogL;
#pragma unroll
  for (int s = 0; s < kSteps; ++s) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, LPP >> (s + 1)));
  return mx;
}

// acc + q0*k0 + q1*k1 for bf16 pairs q = (q0, q1), k = (k0, k1) (low half first): each step is
// one fp32 fma of a bf16 x bf16 product, which is exact in fp32, so the sum is the same as with
// both operands widened to fp32 first. Keeping q as bf16 pairs (32 registers for G = 4) instead
// of fp32 lets four CTAs share an SM.
__device__ __forceinline__ float dot2_bf16(uint32_t q, uint32_t k, float acc) {
  float r;
  asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.bf16 %0, a0, b0, %3;\n fma.rn.f32.bf16 %0, a1, b1, %0;\n}\n"
      : "=f"(r) : "r"(q), "r"(k), "f"(acc));
  return r;
}

// ------------------------------------------------------------------------------------
// page scores, streaming
// ------------------------------------------------------------------------------------
// One CTA per (chunk, sequence, group of up to 8 KV heads): chunks of a.pchunk pages first, then
// each sequence's last a.tail_pages pages in chunks of a.tail_chunk (see launch_t). The summaries of
// a page for the CTA's heads are one contiguous run (H * 2 * D elements; 4 KB at H = 8,
// D = 128 bf16), so warp 0 fetches each page with one bulk copy (TMA engine) into a ring of
// kStages shared-memory stages of a.stage_pages pages, completion tracked by one mbarrier per
// stage (bounded waits). All warps then score from shared memory: warp w takes KV head w % HPC
// of the group and every (8 / HPC)-th page step. Writes one 32-bit order key per page (0 for
// an always-kept page and for pages whose block id is out of range) and, when asked, the fp32
// score.
constexpr int kStages = 2;
constexpr int kStageBytes = 24576;
constexpr int kMaxStagePages = 32;
constexpr int kPageSteps = 1;  // page steps per loop iteration
constexpr int kTailChunk = 16;  // pages per CTA of the tail region
constexpr int kTailWaves = 1;   // resident waves of CTAs that the tail region fills

// kPerQueryHead: the units are the per-query-head view (G = 1 per unit), whose heads share cache
// heads 2^kv_shift at a time; otherwise unit heads are cache heads (a shift of 0 known at compile
// time, which the per-KV-head form is measurably faster with).
template <typename T, int D, int G, bool kPerQueryHead>
__global__ void __launch_bounds__(kThreads, 4) page_score_kernel(ScoreArgs a) {
  pdl_wait();  // the select launch is released at the end of the loop (see below)
  constexpr int EPC = Elem<T>::kPerChunk;
  constexpr int LPP = D / EPC;   // lanes per page
  constexpr int PPW = 32 / LPP;  // pages per warp step
  constexpr int ES = Elem<T>::kBytes;
  static_assert(LPP >= 1 && LPP <= 32 && (LPP & (LPP - 1)) == 0, "row must be 16..512 bytes, power of 2");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kStages];
  __shared__ int okflag[kStages][kMaxStagePages];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kv_shift = kPerQueryHead ? a.kv_shift : 0;
  const int H_cache = kPerQueryHead ? a.H_kv_cache : a.H_kv;
  const int hpc = a.H_kv < kWarps ? a.H_kv : kWarps;  // heads per CTA
  const int ng = kWarps / hpc;                         // warps per head
  // work item of this CTA: (chunk, sequence, head group) with the chunk index fastest, first in
  // the body region (chunks of a.pchunk pages) and then in the tail region (each sequence's last
  // a.tail_pages pages in chunks of a.tail_chunk), so the CTAs dispatched last are short
  int x = blockIdx.x;
  const int n_body = a.body_chunks * a.B * (a.H_kv / hpc);
  const bool in_tail = x >= n_body;
  if (in_tail) x -= n_body;
  const int per_seq = in_tail ? a.tail_chunks : a.body_chunks;
  const int c = x % per_seq;
  x /= per_seq;
  const int i = x % a.B;
  const int h0 = (x / a.B) * hpc;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by the select kernel
  const int body_end = P - min(P, a.tail_pages);
  const int p0 = in_tail ? body_end + c * a.tail_chunk : c * a.pchunk;
  const int p1 = in_tail ? min(P, p0 + a.tail_chunk) : min(body_end, p0 + a.pchunk);
  if (p0 >= p1) return;
  const int hh = warp % hpc;
  const int h = h0 + hh;
  const int wg = warp / hpc;
  const int unit = i * a.H_kv + h;
  // one page's summaries for the CTA's heads: cache heads h0 >> kv_shift .. (h0 + hpc - 1) >> kv_shift
  const int group_bytes = (hpc >> kv_shift) * 2 * D * ES;
  const int sp = a.stage_pages;
  const int n_stages = (p1 - p0 + sp - 1) / sp;
  const T *sumbase = reinterpret_cast<const T *>(a.summaries);
  const int32_t *bt = a.block_table + (size_t)i * a.max_pages;

  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) mbar_init(smem_u32(&bars[k]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // warp 0: block id of this lane's page of stage `st` (-1 past the chunk); loaded one stage
  // ahead of its use so the latency hides behind the current stage's work
  auto block_of = [&](int st) -> int {
    const int p = p0 + st * sp + lane;
    return (lane < sp && st < n_stages && p < p1) ? __ldg(bt + p) : -1;
  };
  // the summaries are read once per step and exceed L2: keep them from evicting what the select
  // and decode kernels read next (keys, selected rows, partials)
  const uint64_t stream_policy = l2_evict_first_policy();
  // warp 0: fetch the pages of stage `st` (chunk-local stage index) into ring slot st % kStages
  auto produce = [&](int st, int blk) {
    const int slot = st % kStages;
    const int p = p0 + st * sp + lane;
    const bool in_chunk = lane < sp && p < p1;
    const bool valid = blk >= 0 && blk < a.nb;
    if (in_chunk && !valid) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    // always-kept pages are kept whatever their score: without scores_out their summaries
    // are not read (so an append to the tail page may run concurrently)
    const bool needed = a.scores_out != nullptr || !always_kept(p, P, a.sink, a.window);
    const bool ok = in_chunk && valid && needed;
    if (lane < sp) okflag[slot][lane] = ok;
    const unsigned mask = __ballot_sync(0xffffffffu, ok);
    const uint32_t bar = smem_u32(&bars[slot]);
    __syncwarp();  // the flags above are ordered before lane 0's release-arrive
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(mask) * group_bytes);
    __syncwarp();
    if (ok)
      bulk_g2s_stream(smem_u32(smem_raw + (size_t)slot * kStageBytes + (size_t)lane * group_bytes),
                      sumbase + ((size_t)blk * H_cache + (h0 >> kv_shift)) * 2 * D, group_bytes, bar, stream_policy);
  };

  if (warp == 0)
    for (int st = 0; st < kStages && st < n_stages; ++st) produce(st, block_of(st));

  const int sub = lane % LPP;  // which 16-byte chunk of the summary row
  const int grp = lane / LPP;  // which page of the warp step
  float2 qp[G][EPC / 2], qn[G][EPC / 2];
  uint32_t qpw[G][4], qnw[G][4];  // bf16 path: max(q,0) / min(q,0) as bf16 pairs (exact)
  {
    const T *qrow = reinterpret_cast<const T *>(a.q) + ((size_t)i * a.H_q + (size_t)h * G) * D + sub * EPC;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint4 w = *reinterpret_cast<const uint4 *>(qrow + (size_t)g * D);
      if constexpr (sizeof(T) == 2) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t m = ((ws[e] & 0x80008000u) >> 15) * 0xFFFFu;  // negative halves
          qnw[g][e] = ws[e] & m;
          qpw[g][e] = ws[e] & ~m;
        }
      } else {
        float2 f[EPC / 2];
        Elem<T>::to_f2(w, f);
#pragma unroll
        for (int e = 0; e < EPC / 2; ++e) {
          qp[g][e] = make_float2(fmaxf(f[e].x, 0.f), fmaxf(f[e].y, 0.f));
          qn[g][e] = make_float2(fminf(f[e].x, 0.f), fminf(f[e].y, 0.f));
        }
      }
    }
  }
  uint32_t *krow = a.keys + (size_t)unit * a.key_stride;
  float *srow = a.scores_out ? a.scores_out + (size_t)unit * a.max_pages : nullptr;
  // this lane's byte offset inside a page's run: its head and its chunk
  const uint32_t lane_off = (uint32_t)(hh >> kv_shift) * 2 * D * ES + sub * 16;

  for (int st = 0; st < n_stages; ++st) {
    const int slot = st % kStages;
    const int next_blk = warp == 0 ? block_of(st + kStages) : -1;  // in flight during this stage
    mbar_wait(smem_u32(&bars[slot]), (st / kStages) & 1, a.ws);
    const unsigned char *stage = smem_raw + (size_t)slot * kStageBytes;
    const int pb = p0 + st * sp;
    const int np = min(sp, p1 - pb);
    // kPageSteps page steps per iteration (all steps' loads first, then independent chains).
    // Loads are unconditional (always inside the stage); pages that are not live (past the
    // chunk, or a flagged block) are dropped when the key is written.
    const uint32_t stage_addr = smem_u32(stage) + lane_off;
    for (int j0 = wg * PPW; j0 < np; j0 += kPageSteps * ng * PPW) {  // warp-uniform bound
      uint4 lo[kPageSteps], hi[kPageSteps];
#pragma unroll
      for (int u = 0; u < kPageSteps; ++u) {
        const int jl = min(j0 + u * ng * PPW + grp, sp - 1);  // stays inside the stage
        const uint32_t addr = stage_addr + (uint32_t)jl * (uint32_t)group_bytes;
        lo[u] = lds128(addr);
        hi[u] = lds128(addr + D * ES);
      }
      float v[kPageSteps][G];
#pragma unroll
      for (int u = 0; u < kPageSteps; ++u) {
        if constexpr (sizeof(T) == 2) {
          const uint32_t kl[4] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w};
          const uint32_t kh[4] = {hi[u].x, hi[u].y, hi[u].z, hi[u].w};
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              a0 = dot2_bf16(qpw[g][e], kh[e], a0);
              a1 = dot2_bf16(qnw[g][e], kl[e], a1);
            }
            v[u][g] = a0 + a1;
          }
        } else {
          float2 kl[EPC / 2], kh[EPC / 2];
          Elem<T>::to_f2(lo[u], kl);
          Elem<T>::to_f2(hi[u], kh);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EPC / 2; ++e) {
              acc = ffma2(qp[g][e], kh[e], acc);
              acc = ffma2(qn[g][e], kl[e], acc);
            }
            v[u][g] = acc.x + acc.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kPageSteps; ++u) {
        const int jb = j0 + u * ng * PPW;
        if (u > 0 && jb >= np) break;  // warp-uniform
        const float sc = group_score<G, LPP>(v[u], lane) * a.scale;
        const int j = jb + grp;
        if (sub == 0 && j < np) {
          const int p = pb + j;
          const bool forced = always_kept(p, P, a.sink, a.window);
          krow[p] = (okflag[slot][j] && !forced) ? score_key(sc) : 0u;
          if (srow) srow[p] = sc;
        }
      }
    }
    __syncthreads();  // every warp is done with this slot
    if (warp == 0 && st + kStages < n_stages) {
      fence_proxy_async_smem();
      produce(st + kStages, next_blk);
    }
  }
  // released here rather than at the start: select CTAs made resident early would sit waiting
  // through this grid's drain
  pdl_trigger();
}

// ------------------------------------------------------------------------------------
// page scores on the tensor cores (bf16 caches, per-KV-head units)
// ------------------------------------------------------------------------------------
// A page's bound for query head g is one dot product of length 2D: its stored summary row
// [kmin | kmax] against [min(q_g,0) | max(q_g,0)] (both halves exact in bf16). So a warp-level
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate) scores 16 (page, KV head) rows at once: rows 0-7
// are 8 consecutive pages of head hA, rows 8-15 8 pages of head hB; columns 0-3 hold hA's query
// heads, columns 4-7 hB's (columns past G are zero). Each row's score is the max over its own
// head's columns; the cross terms are not used. The products are exact in fp32 and the sums are
// fp32 (the tensor cores' order), so the result meets the same bound as the FMA kernel above, at
// 2D / 16 MMAs per 16 rows instead of 2D * G / 16 FMAs per row on each lane.
//
// With G = 8 a head's query heads fill all 8 columns: each MMA takes one KV head, rows 0-7 and
// 8-15 its pages of two consecutive octets.
//
// Staging is the same bulk-copy ring as page_score_kernel with two changes: stages hold a
// multiple of 8 pages, and pages sit group_bytes + 16 bytes apart (group_bytes is a multiple of
// 128), so the 8 rows of an ldmatrix (8 pages of one head, equal offsets inside their rows) fall
// in 8 different bank groups. Warp w takes head pair w % n_pairs of the CTA's heads (one pair
// per two heads, G <= 4: four warps; one head per "pair", G = 8: eight warps; with one head in
// the CTA, or G = 8, rows 8-15 take the next 8 pages of the same head).
template <int G>
__host__ __device__ constexpr int mma_threads() {
  return G > 4 ? 256 : 128;
}
constexpr int kMmaStages = 2;
constexpr int kMmaStageBytes = 32768 + 512;  // 8 pages x (4 KB + 16) at H = 8, D = 128; 32 x (1 KB + 16)

// kPerQueryHead: the units are the per-query-head view (one unit per query head, kv_shift =
// log2 G); the same MMAs run over the cache heads, and each column (query head) is its own unit:
// its score is written as its key, with no max over the group.
template <int D, int G, bool kPerQueryHead = false>
__global__ void __launch_bounds__(mma_threads<G>()) page_score_mma_kernel(ScoreArgs a) {
  pdl_wait();
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "1, 2, 4 or 8 query heads per KV head");
  static_assert(!kPerQueryHead || G > 1, "the per-query-head view groups G > 1 query heads");
  constexpr bool kWide = G > 4;                      // one KV head per MMA
  constexpr int kMmaWarps = mma_threads<G>() / 32;
  constexpr int KS = 2 * D / 16;  // k-steps over a summary row [kmin | kmax]
  constexpr int RB = 2 * D * 2;   // bytes of one (page, head) summary row
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kMmaStages];
  __shared__ int okflag[kMmaStages][kMaxStagePages];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hpc = a.mma_hpc;  // unit heads per CTA (chosen at launch)
  // work item (chunk, sequence, head group): the same order and regions as page_score_kernel
  int x = blockIdx.x;
  const int n_body = a.body_chunks * a.B * (a.H_kv / hpc);
  const bool in_tail = x >= n_body;
  if (in_tail) x -= n_body;
  const int per_seq = in_tail ? a.tail_chunks : a.body_chunks;
  const int c = x % per_seq;
  x /= per_seq;
  const int i = x % a.B;
  const int h0 = (x / a.B) * hpc;
  // cache heads of the CTA: per KV head, the unit heads themselves; per query head, the unit heads
  // h0 .. h0 + hpc - 1 read cache heads h0 / G .. (h0 + hpc - 1) / G
  const int hcc = kPerQueryHead ? hpc / G : hpc;
  const int hc0 = kPerQueryHead ? h0 / G : h0;
  const int H_cache = kPerQueryHead ? a.H_kv_cache : a.H_kv;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by the select kernel
  const int body_end = P - min(P, a.tail_pages);
  const int p0 = in_tail ? body_end + c * a.tail_chunk : c * a.pchunk;
  const int p1 = in_tail ? min(P, p0 + a.tail_chunk) : min(body_end, p0 + a.pchunk);
  if (p0 >= p1) return;
  const int group_bytes = hcc * RB;
  const int sp = a.stage_pages;  // a multiple of 8
  const int n_stages = (p1 - p0 + sp - 1) / sp;
  const bf16_t *sumbase = reinterpret_cast<const bf16_t *>(a.summaries);
  const int32_t *bt = a.block_table + (size_t)i * a.max_pages;

  if (tid == 0) {
    for (int k = 0; k < kMmaStages; ++k) mbar_init(smem_u32(&bars[k]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto block_of = [&](int st) -> int {
    const int p = p0 + st * sp + lane;
    return (lane < sp && st < n_stages && p < p1) ? __ldg(bt + p) : -1;
  };
  const uint64_t stream_policy = l2_evict_first_policy();
  auto produce = [&](int st, int blk) {
    const int slot = st % kMmaStages;
    const int p = p0 + st * sp + lane;
    const bool in_chunk = lane < sp && p < p1;
    const bool valid = blk >= 0 && blk < a.nb;
    if (in_chunk && !valid) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    const bool needed = a.scores_out != nullptr || !always_kept(p, P, a.sink, a.window);
    const bool ok = in_chunk && valid && needed;
    if (lane < sp) okflag[slot][lane] = ok;
    const unsigned mask = __ballot_sync(0xffffffffu, ok);
    const uint32_t bar = smem_u32(&bars[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(mask) * group_bytes);
    __syncwarp();
    if (ok)
      bulk_g2s_stream(smem_u32(smem_raw + (size_t)slot * kMmaStageBytes + (size_t)lane * (group_bytes + 16)),
                      sumbase + ((size_t)blk * H_cache + hc0) * 2 * D, group_bytes, bar, stream_policy);
  };

  if (warp == 0)
    for (int st = 0; st < kMmaStages && st < n_stages; ++st) produce(st, block_of(st));

  // head pair of this warp (heads local to the CTA's group); G = 8: one head
  const int n_pairs = kWide ? hcc : (hcc >= 2 ? hcc / 2 : 1);
  const int pair = warp % n_pairs, wsub = warp / n_pairs, wpp = kMmaWarps / n_pairs;
  const int hlA = kWide ? pair : (hcc >= 2 ? 2 * pair : 0);
  const int hlB = kWide ? pair : (hcc >= 2 ? 2 * pair + 1 : 0);
  const bool octet_pairs = kWide || hcc == 1;  // rows 8-15: the next 8 pages of the same head

  // B fragments for all k-steps: lane holds column n = lane / 4 (head hA for n < 4, else hB;
  // query head n % 4 of it; G = 8: query head n of the warp's head) at k = 2t, 2t+1 (b0) and
  // 2t+8, 2t+9 (b1) of each k-step, t = lane % 4. k-steps 0 .. D/16-1 meet kmin (min(q,0)), the
  // rest kmax (max(q,0)).
  uint32_t bq[KS][2];
  {
    const int n = lane >> 2, t = lane & 3;
    const int g = kWide ? n : (n & 3);
    const int hl = (kWide || n < 4) ? hlA : hlB;
    if (g < G) {
      const uint32_t *qr = reinterpret_cast<const uint32_t *>(reinterpret_cast<const bf16_t *>(a.q) +
                                                              ((size_t)i * a.H_q + (size_t)(hc0 + hl) * G + g) * D);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t w = __ldg(qr + 8 * s + t + 4 * e);
          const uint32_t m = ((w & 0x80008000u) >> 15) * 0xFFFFu;  // negative halves
          bq[s][e] = w & m;               // min(q, 0)
          bq[s + D / 16][e] = w & ~m;     // max(q, 0)
        }
      }
    } else {
#pragma unroll
      for (int s = 0; s < KS; ++s) bq[s][0] = bq[s][1] = 0u;
    }
  }

  // ldmatrix row of this lane: matrix mi = lane / 8 (rows 0-7 or 8-15, k 0-7 or 8-15 of the step)
  const int mi = lane >> 3, rr = lane & 7;
  const bool rowB = (mi & 1) != 0;
  const uint32_t lane_off = (uint32_t)(rowB ? hlB : hlA) * RB + (uint32_t)(mi >> 1) * 16;
  // epilogue position: rows r0 (item A) / r0 + 8 (item B), columns 2t, 2t + 1
  const int r0 = lane >> 2, t = lane & 3;
  const bool outB = t >= 2;
  const int g0 = 2 * (t & 1);

  for (int st = 0; st < n_stages; ++st) {
    const int slot = st % kMmaStages;
    const int next_blk = warp == 0 ? block_of(st + kMmaStages) : -1;
    mbar_wait(smem_u32(&bars[slot]), (st / kMmaStages) & 1, a.ws);
    const uint32_t stage_addr = smem_u32(smem_raw + (size_t)slot * kMmaStageBytes);
    const int pb = p0 + st * sp;
    const int np = min(sp, p1 - pb);
    const int n_oct = (np + 7) >> 3;
    const int n_items = octet_pairs ? (n_oct + 1) >> 1 : n_oct;
    for (int m = wsub; m < n_items; m += wpp) {  // warp-uniform bound
      const int oA = octet_pairs ? 2 * m : m, oB = octet_pairs ? 2 * m + 1 : m;
      // rows past the stage's live pages read the last page of the stage (discarded below)
      const int j = min(((rowB ? oB : oA) << 3) + rr, sp - 1);
      const uint32_t addr = stage_addr + (uint32_t)j * (uint32_t)(group_bytes + 16) + lane_off;
      float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < KS; s += 2) {
        uint32_t fa[4], fb[4];
        ldsm_x4(addr + s * 32, fa);
        ldsm_x4(addr + s * 32 + 32, fb);
        mma_16816_bf16(acc0, fa, bq[s][0], bq[s][1]);
        mma_16816_bf16(acc1, fb, bq[s + 1][0], bq[s + 1][1]);
      }
      if constexpr (kPerQueryHead) {
        // every column is a unit. G <= 4: lane (r0, t) holds columns 2t, 2t + 1 of row r0 (head
        // A) for t < 2, of row r0 + 8 (head B) for t >= 2. G = 8: columns 2t, 2t + 1 of rows r0
        // and r0 + 8 (two octets of the same head).
        auto put = [&](int oct, int hl, int g, float v) {
          const int jo = (oct << 3) + r0;
          if (g < G && jo < np) {
            const int p = pb + jo;
            const int unit = i * a.H_kv + (hc0 + hl) * G + g;
            const float sc = v * a.scale;
            const bool forced = always_kept(p, P, a.sink, a.window);
            a.keys[(size_t)unit * a.key_stride + p] = (okflag[slot][jo] && !forced) ? score_key(sc) : 0u;
            if (a.scores_out) a.scores_out[(size_t)unit * a.max_pages + p] = sc;
          }
        };
        const float v0 = acc0[0] + acc1[0], v1 = acc0[1] + acc1[1];
        const float v2 = acc0[2] + acc1[2], v3 = acc0[3] + acc1[3];
        if constexpr (kWide) {
          put(oA, hlA, 2 * t, v0);
          put(oA, hlA, 2 * t + 1, v1);
          put(oB, hlA, 2 * t, v2);
          put(oB, hlA, 2 * t + 1, v3);
        } else {
          put(outB ? oB : oA, outB ? hlB : hlA, g0, outB ? v2 : v0);
          put(outB ? oB : oA, outB ? hlB : hlA, g0 + 1, outB ? v3 : v1);
        }
      } else if constexpr (kWide) {
        // row r0 (octet oA) and row r0 + 8 (octet oB) of the warp's head, columns 2t, 2t + 1 of
        // its 8 query heads: the max over the 8 columns takes two shuffles per row
        float vA = fmaxf(acc0[0] + acc1[0], acc0[1] + acc1[1]);
        float vB = fmaxf(acc0[2] + acc1[2], acc0[3] + acc1[3]);
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          vA = fmaxf(vA, __shfl_xor_sync(0xffffffffu, vA, o));
          vB = fmaxf(vB, __shfl_xor_sync(0xffffffffu, vB, o));
        }
        if (t == 0) {
          const int unit = i * a.H_kv + hc0 + hlA;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int jo = ((r ? oB : oA) << 3) + r0;
            if (jo < np) {
              const int p = pb + jo;
              const float sc = (r ? vB : vA) * a.scale;
              const bool forced = always_kept(p, P, a.sink, a.window);
              a.keys[(size_t)unit * a.key_stride + p] = (okflag[slot][jo] && !forced) ? score_key(sc) : 0u;
              if (a.scores_out) a.scores_out[(size_t)unit * a.max_pages + p] = sc;
            }
          }
        }
      } else {
        const float x0 = outB ? acc0[2] + acc1[2] : acc0[0] + acc1[0];
        const float x1 = outB ? acc0[3] + acc1[3] : acc0[1] + acc1[1];
        float v = g0 < G ? x0 : -INFINITY;
        if (g0 + 1 < G) v = fmaxf(v, x1);
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
        const int jo = ((outB ? oB : oA) << 3) + r0;
        if ((t & 1) == 0 && jo < np) {
          const int p = pb + jo;
          const int unit = i * a.H_kv + hc0 + (outB ? hlB : hlA);
          const float sc = v * a.scale;
          const bool forced = always_kept(p, P, a.sink, a.window);
          a.keys[(size_t)unit * a.key_stride + p] = (okflag[slot][jo] && !forced) ? score_key(sc) : 0u;
          if (a.scores_out) a.scores_out[(size_t)unit * a.max_pages + p] = sc;
        }
      }
    }
    __syncthreads();  // every warp is done with this slot
    if (warp == 0 && st + kMmaStages < n_stages) {
      fence_proxy_async_smem();
      produce(st + kMmaStages, next_blk);
    }
  }
  pdl_trigger();
}

// The score kernel for these units: the tensor-core kernel for bf16 caches (unless
// PSK_SCORE_MMA=0), per KV head or per query head, else the FMA kernel. G = 8 is built on the
// tensor cores only.
enum class ScoreKernel { kFma, kFmaPerQueryHead, kMma, kMmaPerQueryHead };

template <int D, int Gc>
cudaError_t launch_mma_pqh(unsigned n_ctas, int smem, cudaStream_t s, const ScoreArgs &b) {
  return launch_kernel(true, page_score_mma_kernel<D, Gc, true>, n_ctas, mma_threads<Gc>(), smem, s, b);
}

template <typename T, int D, int G>
const void *score_kernel_fn(ScoreKernel k, int kv_shift) {
  if constexpr (sizeof(T) == 2) {
    if (k == ScoreKernel::kMma) return reinterpret_cast<const void *>(page_score_mma_kernel<D, G>);
    if constexpr (G == 1) {
      if (k == ScoreKernel::kMmaPerQueryHead) {
        if (kv_shift == 1) return reinterpret_cast<const void *>(page_score_mma_kernel<D, 2, true>);
        if (kv_shift == 2) return reinterpret_cast<const void *>(page_score_mma_kernel<D, 4, true>);
        if (kv_shift == 3) return reinterpret_cast<const void *>(page_score_mma_kernel<D, 8, true>);
        return nullptr;
      }
    }
  }
  if constexpr (G <= 4) {
    if (k == ScoreKernel::kFmaPerQueryHead) return reinterpret_cast<const void *>(page_score_kernel<T, D, G, true>);
    if (k == ScoreKernel::kFma) return reinterpret_cast<const void *>(page_score_kernel<T, D, G, false>);
  }
  return nullptr;
}

template <typename T, int D, int G>
cudaError_t launch_t(const ScoreArgs &a, cudaStream_t s, int stages) {
  if (!(stages & kStageScore)) return launch_page_select(a, s, true);
  if (G > 1 && a.kv_shift != 0) return cudaErrorInvalidValue;  // the per-query-head view has G = 1
  int hpc = a.H_kv < kWarps ? a.H_kv : kWarps;  // unit heads per CTA
  ScoreArgs b = a;
  ScoreKernel kind = a.kv_shift != 0 ? ScoreKernel::kFmaPerQueryHead : ScoreKernel::kFma;
  int threads = kThreads;
  int smem = kStages * kStageBytes;
  if (sizeof(T) == 2 && a.kv_shift <= 3 && (tuning().score_mma || G > 4)) {
    kind = a.kv_shift != 0 ? ScoreKernel::kMmaPerQueryHead : ScoreKernel::kMma;
    threads = a.kv_shift == 3 || G > 4 ? 256 : 128;  // mma_threads of the cache group size
    smem = kMmaStages * kMmaStageBytes;
    if (a.kv_shift != 0) {  // per query head: 8 cache heads' query heads when they divide the units
      const int wide = std::min(a.H_kv, kWarps << a.kv_shift);
      if (a.H_kv % wide == 0) hpc = wide;
    }
    b.mma_hpc = hpc;
    const int group_bytes = (hpc >> a.kv_shift) * 2 * D * 2;  // <= 4 KB, so at least 8 pages per stage
    b.stage_pages = std::min(kMaxStagePages, kMmaStageBytes / (group_bytes + 16)) / 8 * 8;
  }
  const void *fn = score_kernel_fn<T, D, G>(kind, a.kv_shift);
  if (!fn) return cudaErrorInvalidValue;
  // Tail region: about kTailWaves waves of short CTAs over the sequences' last pages. A grid of
  // equal chunks ends with its last wave draining for one whole CTA lifetime at falling
  // occupancy; short CTAs last make that drain short.
  {
    int per_sm = 0;
    cudaError_t e = kernel_setup(fn, threads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    const Tuning &tu = tuning();
    b.tail_chunk = tu.score_tail_chunk > 0 ? tu.score_tail_chunk : kTailChunk;
    const long long rows = (long long)a.B * (a.H_kv / hpc);
    long long tail = ((long long)sm_count() * std::max(1, per_sm) * kTailChunk * kTailWaves + rows - 1) / rows;
    if (tu.score_tail >= 0) tail = tu.score_tail;  // tuning override: pages
    tail = (tail + b.tail_chunk - 1) / b.tail_chunk * b.tail_chunk;
    b.tail_pages = (int)std::max(0LL, std::min(tail, (long long)a.max_pages));
    b.tail_chunks = (b.tail_pages + b.tail_chunk - 1) / b.tail_chunk;
    b.body_chunks = (a.max_pages + a.pchunk - 1) / a.pchunk;
  }
  const long long n_ctas = (long long)(b.body_chunks + b.tail_chunks) * b.B * (b.H_kv / hpc);
  if (n_ctas > INT32_MAX) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaErrorInvalidValue;
  if (kind == ScoreKernel::kMma) {
    if constexpr (sizeof(T) == 2)
      e = launch_kernel(true, page_score_mma_kernel<D, G>, (unsigned)n_ctas, threads, smem, s, b);
  } else if (kind == ScoreKernel::kMmaPerQueryHead) {
    if constexpr (sizeof(T) == 2 && G == 1) {
      if (a.kv_shift == 1) e = launch_mma_pqh<D, 2>((unsigned)n_ctas, smem, s, b);
      if (a.kv_shift == 2) e = launch_mma_pqh<D, 4>((unsigned)n_ctas, smem, s, b);
      if (a.kv_shift == 3) e = launch_mma_pqh<D, 8>((unsigned)n_ctas, smem, s, b);
    }
  } else if constexpr (G <= 4) {
    if (kind == ScoreKernel::kFmaPerQueryHead) {
      if constexpr (G == 1)
        e = launch_kernel(true, page_score_kernel<T, D, G, true>, (unsigned)n_ctas, threads, smem, s, b);
    } else {
      e = launch_kernel(true, page_score_kernel<T, D, G, false>, (unsigned)n_ctas, threads, smem, s, b);
    }
  }
  if (e != cudaSuccess || !(stages & kStageSelect)) return e;
  return launch_page_select(b, s);
}

}  // namespace

bool plan_score(const psk_layout &L, int b_max, ScorePlan *plan, int kv_shift) {
  if (L.num_kv_heads > kWarps && L.num_kv_heads % kWarps != 0) return false;
  if (L.num_kv_heads < kWarps && kWarps % L.num_kv_heads != 0) return false;
  const int kfree_max = std::max(1, b_max - 1);  // at least the tail page is always kept
  int chunk = 4096;
  if (tuning().select_chunk > 0) chunk = tuning().select_chunk;  // tuning override: pages per selection CTA
  while (true) {
    const int nch = (L.max_pages + chunk - 1) / chunk;
    const int kcap = std::min(kfree_max, chunk);
    if (nch == 1 || (long long)nch * kcap <= kMergeCap) break;
    chunk *= 2;
    if (chunk > 16384) return false;
  }
  plan->chunk = chunk;
  plan->n_chunks_max = (L.max_pages + chunk - 1) / chunk;
  plan->k_cap = std::min(kfree_max, chunk);
  // pages per streaming CTA of the body region: 64 (measured best on the batched workload, 48,
  // 96 and 128 slower); fewer only while the body would not fill one resident wave (four CTAs on
  // each SM), since the tail region supplies the short CTAs at the end (one 1M-token sequence:
  // 64 pages 62.9 us against 66.2 us at 32)
  const long long head_groups = L.num_kv_heads > kWarps ? L.num_kv_heads / kWarps : 1;
  int pchunk = 64;
  const long long wave = 4LL * sm_count();
  while (pchunk > 16 && (long long)L.batch * head_groups * ((L.max_pages + pchunk - 1) / pchunk) < wave)
    pchunk /= 2;
  if (tuning().score_pchunk > 0) pchunk = tuning().score_pchunk;  // tuning override: pages per score CTA
  plan->pchunk = pchunk;
  {
    const int hpc = L.num_kv_heads < kWarps ? L.num_kv_heads : kWarps;
    const int es = L.dtype == PSK_F32 ? 4 : 2;
    const int group_bytes = (hpc >> kv_shift) * 2 * L.head_dim * es;
    plan->stage_pages = group_bytes > kStageBytes ? 1 : std::min(kMaxStagePages, kStageBytes / group_bytes);
    if (group_bytes > kStageBytes && !L.latent) return false;
  }
  const size_t units = (size_t)L.batch * L.num_kv_heads;
  plan->off_counters = ws_score_tickets_offset();
  size_t off = ws_scratch_offset(units);
  plan->off_keys = off;
  off = align_up(off + units * (size_t)((L.max_pages + 3) & ~3) * 4, 256);
  plan->off_key = off;
  off = align_up(off + units * plan->n_chunks_max * plan->k_cap * 4, 256);
  plan->off_page = off;
  off = align_up(off + units * plan->n_chunks_max * plan->k_cap * 4, 256);
  plan->off_count = off;
  off = align_up(off + units * plan->n_chunks_max * 4, 256);
  plan->off_qsplit = off;
  if (L.latent) off = align_up(off + mla_qsplit_bytes(L), 256);
  plan->ws_bytes = off;
  return true;
}

#define PSK_SCORE_CASES(X)   \
  X(bf16_t, PSK_BF16, 128, 4) \
  X(bf16_t, PSK_BF16, 128, 8) \
  X(bf16_t, PSK_BF16, 64, 4)  \
  X(float, PSK_F32, 64, 4)    \
  X(float, PSK_F32, 128, 4)   \
  X(bf16_t, PSK_BF16, 128, 1) \
  X(bf16_t, PSK_BF16, 128, 2) \
  X(bf16_t, PSK_BF16, 64, 1)  \
  X(bf16_t, PSK_BF16, 64, 2)  \
  X(float, PSK_F32, 64, 1)    \
  X(float, PSK_F32, 128, 1)

bool score_supported(int dtype, int D, int G) {
#define X(TT, DT, DD, GG) \
  if (dtype == DT && D == DD && G == GG) return true;
  PSK_SCORE_CASES(X)
#undef X
  return false;
}

cudaError_t launch_score_select(const ScoreArgs &a, int dtype, cudaStream_t s, int stages) {
  const int D = a.D, G = a.H_q / a.H_kv;
#define X(TT, DT, DD, GG) \
  if (dtype == DT && D == DD && G == GG) return launch_t<TT, DD, GG>(a, s, stages);
  PSK_SCORE_CASES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace psk
