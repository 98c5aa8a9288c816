// Stage 4: exact softmax attention over the selected pages of a GQA paged cache, split-K over
// pages with an fp32 online-softmax (m, l, O) state and a log-sum-exp merge (EntmaxKV README,
// introduction: "the attention is exact over that selection"; LOCKS PKG-INFO, "How it works",
// Sparse decode: a paged kernel that reads only the selected pages). The dense decode is the
// same kernel with the implicit page list 0 .. P-1.
//
// Work: one CTA of NW warps (4; 8 when the grid is smaller than one CTA per SM) per (split of
// `sw` list entries, KV head, sequence). The group's G
// query heads share every K/V element loaded, so each element is converted once and used G
// times. A page is cut into 16-token tiles; warp w takes tiles w, w + NW, ... of the split and
// keeps its own (m, l, O) state. Lane 0 of each warp stages the tiles into the warp's ring of
// NST shared-memory stages with 3-D TMA copies (K and V, box D x 1 head x 16 rows, L2
// evict-first), completing on the stage's mbarrier, NST - 1 tiles in flight per warp. Rows past
// seq_len may hold anything: their logits are masked to -inf and P.V stops at the last valid row.
//
// FMA tiles (fp32 caches; bf16 when PSK_DECODE_MMA=0), per tile and warp: lane = (tq = lane / 8,
// dg = lane % 8). QK: the lane owns the 16-byte
// chunks dg, dg + 8, ... of each K row and the matching q slices (scaled by scale * log2(e) so
// exp2 gives the softmax weights) and computes partial dot products for tokens tq, tq + 4,
// tq + 8, tq + 12 and all G heads with packed fp32x2 FMAs; a transposing butterfly over the 8
// dg lanes leaves each lane the full logits of one token for G/2 heads. Online softmax: tile
// max per head by 4 shuffles, rescale only when the max moved, p to a per-warp array as (p, p)
// pairs. PV: the lane owns D/32 output dims of all G heads and accumulates with packed FMAs
// from one conflict-free V row chunk per token.
//
// bf16 caches compute each tile on the tensor cores instead (warp_tiles_mma over an MmaWarp
// state; the default, and the only form for G = 8): S = q K^T and O += P V as warp-level
// m16n8k16 MMAs (bf16 in, fp32 accumulate), with the query heads as the M rows. The tiles then arrive as 128-byte TMA boxes stored with the 128-byte
// swizzle, so ldmatrix reads K (as is) and V (transposed) without bank conflicts. P stays in
// registers: its fp32 weights are split into a bf16 high part (rows 0..7 of the A fragment)
// and the bf16 rounding of the remainder (rows 8..15, otherwise unused), so P V carries about
// 16 bits of each weight, and the two halves of O are added at the end.
//
// The NW warp states are merged through shared memory into one partial per CTA (m, l and O
// relative to m). Every CTA of a (sequence, KV head) then takes a ticket (CTAs without pages
// write an empty partial first); the CTA holding the last ticket (no waiting) merges the
// unit's partials by log-sum-exp with all its threads and writes the G output rows.
#include <algorithm>

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSwMax = 256;    // list entries per split, upper bound
constexpr int kMaxItems = 256; // splits per (sequence, KV head), upper bound (bounds the merge)
constexpr int kFlatMaxCtas = 2048;   // grid of the flat layout, upper bound (sizes the partials)
constexpr int kFlatMaxUnits = 4096;  // units the flat layout takes (its prefix sums live in shared memory)
constexpr long long kFlatMinShare = 8;  // list entries per CTA of the flat layout, lower bound
constexpr int kFastMerge = 16;         // partials a unit merge reads in one round trip
constexpr int kHostPrefetch = 2;       // host value path: tiles of its own a warp prefetches ahead into L2

template <typename T, int D, int G, int NW, int NST>
struct DT {
  static constexpr int ES = Elem<T>::kBytes;
  static constexpr int EPC = Elem<T>::kPerChunk;  // elements per 16-byte chunk
  static constexpr int NC = D / EPC;               // chunks per row
  static constexpr int CPL = NC / 8;               // QK chunks per lane
  static constexpr int VPL = D / 32;               // PV dims per lane
  static constexpr int ROW = D * ES;               // bytes per row
  static constexpr int TILE = 16 * ROW;
  static constexpr int STAGE = 2 * TILE;           // K tile + V tile
  static constexpr int NV = 4 * G;                 // partial logits per lane before reduce
  static constexpr int KEEP = NV >= 8 ? NV / 8 : 1;
  static constexpr size_t STAGES = (size_t)NW * NST * STAGE;
  static constexpr size_t SMEM = 1024                          // alignment slack (swizzled TMA boxes)
                                 + STAGES                      // stages (reused by the merges)
                                 + (size_t)NW * 16 * G * 8     // (p, p) pairs
                                 + (size_t)NW * G * 2 * 4      // warp m, l
                                 + (size_t)kSwMax * 3 * 4;     // entry table
  static_assert(STAGES >= (size_t)NW * G * D * 4, "stage memory must hold the warps' O for the CTA merge");
  static_assert(NC % 8 == 0, "a row must be a multiple of 128 bytes");
  static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
};

// Transposing reduction over the 8 lanes that differ in lane bits 0..2.
template <int NV>
__device__ __forceinline__ void reduce_dg(float (&v)[NV], int lane) {
  int L = NV;
#pragma unroll
  for (int mask = 4; mask >= 1; mask >>= 1) {
    if (L > 1) {
      const int half = L / 2;
      const bool upper = (lane & mask) != 0;
#pragma unroll
      for (int k = 0; k < NV / 2; ++k) {
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
}

// The last CTA of a unit: merge its n partials (m, l, O) at slots it0 .. it0 + n - 1 by
// log-sum-exp into the G output rows.
// wsm: >= n * G floats of shared memory; red: >= 2 * G * NW floats.
template <typename T, int D, int G, int NW, bool kFast>
__device__ void merge_unit(const DecodeArgs &a, int unit, size_t it0, int n, float *wsm, float *red) {
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (kFast && n <= kFastMerge) {
    // Few partials: every thread reads the (m, l) of its head from all of them together with its
    // O elements (independent loads, one round trip) and merges on its own, without barriers.
    T *out = reinterpret_cast<T *>(a.out) + ((size_t)(unit / a.H_kv) * a.H_q + (size_t)(unit % a.H_kv) * G) * D;
#pragma unroll 1
    for (int idx = tid; idx < G * D; idx += NT) {
      const int g = idx / D;
      float mk[kFastMerge], lk[kFastMerge], ok[kFastMerge];
#pragma unroll
      for (int k = 0; k < kFastMerge; ++k)
        if (k < n) {
          mk[k] = __ldcg(a.part_ml + ((it0 + k) * G + g) * 2);
          lk[k] = __ldcg(a.part_ml + ((it0 + k) * G + g) * 2 + 1);
          ok[k] = __ldcg(a.part_o + (it0 + k) * G * D + idx);
        }
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kFastMerge; ++k)
        if (k < n) M = fmaxf(M, mk[k]);
      float acc = 0.f, L = 0.f;
#pragma unroll
      for (int k = 0; k < kFastMerge; ++k)
        if (k < n && mk[k] != -INFINITY) {
          const float w = exp2f(mk[k] - M);
          acc = fmaf(w, ok[k], acc);
          L = fmaf(w, lk[k], L);
        }
      Elem<T>::store(out + idx, L > 0.f ? acc / L : 0.f);
    }
    return;
  }
  // 1. per-head max of m over the partials
  float mx[G];
#pragma unroll
  for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
  for (int s = tid; s < n; s += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m = __ldcg(a.part_ml + ((it0 + s) * G + g) * 2);
      wsm[s * G + g] = m;
      mx[g] = fmaxf(mx[g], m);
    }
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
    if (lane == 0) red[warp * G + g] = mx[g];
  }
  __syncthreads();
  float M[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = red[g];
#pragma unroll
    for (int w = 1; w < NW; ++w) M[g] = fmaxf(M[g], red[w * G + g]);
  }
  // 2. weights and the normaliser
  float lsum[G];
#pragma unroll
  for (int g = 0; g < G; ++g) lsum[g] = 0.f;
  for (int s = tid; s < n; s += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m = wsm[s * G + g];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M[g]);
      wsm[s * G + g] = w;
      if (w > 0.f) lsum[g] = fmaf(w, __ldcg(a.part_ml + ((it0 + s) * G + g) * 2 + 1), lsum[g]);
    }
  __syncthreads();  // everyone has read red[] before it is reused
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], o);
    if (lane == 0) red[NW * G + warp * G + g] = lsum[g];
  }
  __syncthreads();
  // 3. weighted sum of the partial O rows; thread owns elements tid, tid + NT, ... of [G][D]
  T *out = reinterpret_cast<T *>(a.out) + ((size_t)(unit / a.H_kv) * a.H_q + (size_t)(unit % a.H_kv) * G) * D;
  for (int idx = tid; idx < G * D; idx += NT) {
    const int g = idx / D;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) L += red[NW * G + w * G + g];
    float acc0 = 0.f, acc1 = 0.f;
    int s = 0;
    for (; s + 1 < n; s += 2) {
      const float w0 = wsm[s * G + g], w1 = wsm[(s + 1) * G + g];
      const float o0 = __ldcg(a.part_o + (it0 + s) * G * D + idx);
      const float o1 = __ldcg(a.part_o + (it0 + s + 1) * G * D + idx);
      acc0 = fmaf(w0, w0 > 0.f ? o0 : 0.f, acc0);
      acc1 = fmaf(w1, w1 > 0.f ? o1 : 0.f, acc1);
    }
    if (s < n) {
      const float w0 = wsm[s * G + g];
      const float o0 = __ldcg(a.part_o + (it0 + s) * G * D + idx);
      acc0 = fmaf(w0, w0 > 0.f ? o0 : 0.f, acc0);
    }
    Elem<T>::store(out + idx, L > 0.f ? (acc0 + acc1) / L : 0.f);
  }
}

// List entries [e0, e0 + n) of unit (i, h) (selected row, or pages e0.. when dense) into the
// entry table: physical block and live rows (0 for padding and for flagged entries). All
// threads of the CTA take part; the caller synchronises.
template <int NT>
__device__ void load_entries(const DecodeArgs &a, int i, int unit, int P, int seq_len, int e0, int n, int *ent_blk,
                             int *ent_valid, int *ent_vslot = nullptr) {
  for (int x = threadIdx.x; x < n; x += NT) {
    int p = e0 + x, blk = -1;
    bool ok = true;
    if (a.selected) {
      const int32_t *row = a.selected + (size_t)unit * a.b_max;
      p = row[e0 + x];
      const int prev = (e0 + x > 0) ? row[e0 + x - 1] : -1;
      if (p >= 0 && (p >= P || p <= prev || (e0 + x > 0 && prev < 0))) {
        set_status(a.ws, PSK_DEV_BAD_SELECTED);
        ok = false;
      }
      if (p < 0) ok = false;  // padding
    }
    if (ok) {
      blk = a.block_table[(size_t)i * a.max_pages + p];
      if (blk < 0 || blk >= a.nb) {
        set_status(a.ws, PSK_DEV_BAD_BLOCK);
        ok = false;
      }
    }
    ent_blk[x] = blk;
    ent_valid[x] = ok ? min(a.ps, seq_len - p * a.ps) : 0;
    if (ent_vslot) {
      // a resident copy serves only full pages below the tail (the tail page still takes appends)
      int slot = -1;
      if (ok && a.v_slot && p < P - 1) {
        const int hc = (unit % a.H_kv) >> a.kv_shift;
        slot = a.v_slot[((size_t)i * a.H_kv_cache + hc) * a.max_pages + p];
        if (slot >= a.n_slots) {
          set_status(a.ws, PSK_DEV_BAD_SELECTED);
          slot = -1;
        }
      }
      ent_vslot[x] = slot;
    }
  }
}

// Query slices of this lane (chunks dg, dg + 8, ... of each of the G rows), scaled into the log2
// domain.
template <typename T, int D, int G, int NW, int NST>
__device__ __forceinline__ void load_q(const DecodeArgs &a, int i, int h, int dg,
                                       float2 (&q2)[G][DT<T, D, G, NW, NST>::CPL * DT<T, D, G, NW, NST>::EPC / 2]) {
  using TR = DT<T, D, G, NW, NST>;
  const T *qb = reinterpret_cast<const T *>(a.q) + ((size_t)i * a.H_q + (size_t)h * G) * D;
  const float qs = a.scale * kLog2e;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int c = 0; c < TR::CPL; ++c) {
      float2 f[TR::EPC / 2];
      Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(qb + (size_t)g * D + (dg + 8 * c) * TR::EPC), f);
#pragma unroll
      for (int e = 0; e < TR::EPC / 2; ++e) q2[g][c * TR::EPC / 2 + e] = make_float2(f[e].x * qs, f[e].y * qs);
    }
}

// Value tier: this lane's 8-byte slice (dims lane * 4 ..) of the V rows of tile `it` of the
// entry table, rows at or past the tile's live rows zero. A row comes from the page's resident
// HBM slot when it has one, else from the host cache over NVLink-C2C. The host rows of tile
// it + kHostPrefetch * nw are first prefetched into L2 (one 128-byte line per lane, two lanes
// per row), so their C2C latency overlaps this tile. Built for bf16, D = 128.
template <typename T, int D>
__device__ __forceinline__ void host_v_rows(const DecodeArgs &a, int h, int it, int ntiles, int nw, int stp,
                                            const int *ent_blk, const int *ent_valid, const int *ent_vslot,
                                            uint2 (&vh)[16]) {
  static_assert(D / 32 * sizeof(T) == 8, "8 bytes of V per lane and row");
  const int lane = threadIdx.x & 31;
  auto rows_of = [&](int x) -> int {
    const int e = stp == 1 ? x : x / stp, sub = x - e * stp;
    return min(16, ent_valid[e] - sub * 16);
  };
  auto vsrc = [&](int x, size_t *stride) -> const T * {
    const int e = stp == 1 ? x : x / stp, sub = x - e * stp;
    const int slot = ent_vslot ? ent_vslot[e] : -1;
    if (slot >= 0) {
      *stride = D;
      return reinterpret_cast<const T *>(a.v_hot) + ((size_t)slot * a.ps + sub * 16) * D;
    }
    *stride = (size_t)a.H_kv_cache * D;
    return reinterpret_cast<const T *>(a.v_cache) +
           (((size_t)ent_blk[e] * a.ps + sub * 16) * a.H_kv_cache + (h >> a.kv_shift)) * D;
  };
  const int pf = it + kHostPrefetch * nw;
  if (pf < ntiles && rows_of(pf) > 0) {
    size_t st;
    const T *pb = vsrc(pf, &st);
    if ((lane >> 1) < rows_of(pf))
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(pb + (size_t)(lane >> 1) * st + (lane & 1) * 64) : "memory");
  }
  const int nvh = rows_of(it);
  size_t st;
  const T *vb = vsrc(it, &st) + lane * (D / 32);
#pragma unroll
  for (int tk = 0; tk < 16; ++tk)  // only rows below seq_len: the rest may hold anything
    vh[tk] = tk < nvh ? *reinterpret_cast<const uint2 *>(vb + (size_t)tk * st) : make_uint2(0u, 0u);
}

// Streams the 16-token tiles of the n_ent entries in the entry table through this warp's TMA
// ring (warp w takes tiles w, w + NW, ...) and folds them into the warp's (m, l, O). cw is the
// warp's running tile count: ring stage and mbarrier phase carry on across calls. q_seq >= 0:
// q2 is loaded here (sequence q_seq), after the first tiles' copies are issued, so that its
// global load overlaps their latency; q_seq < 0: the caller has loaded q2.
// kHostV: V rows live in host memory the GPU reads over NVLink-C2C through unified addressing
// (the value tier); only K goes through the TMA ring, and each lane loads its own V slice of
// the tile's valid rows with plain loads when the tile starts, so the C2C latency overlaps the
// QK product and the softmax. Built for 8 bytes of V per lane and row (bf16, D = 128).
template <typename T, int D, int G, int NW, int NST, bool kHostV = false>
__device__ __forceinline__ void warp_tiles(const DecodeArgs &a, const CUtensorMap *tmK, const CUtensorMap *tmV, int h,
                                           int q_seq,
                                           float2 (&q2)[G][DT<T, D, G, NW, NST>::CPL * DT<T, D, G, NW, NST>::EPC / 2],
                                           const int *ent_blk, const int *ent_valid, int n_ent, unsigned char *stages,
                                           float2 *pp_all, uint64_t (*bars)[NST], int &cw, float (&m)[G], float (&l)[G],
                                           float2 (&O)[G][DT<T, D, G, NW, NST>::VPL / 2],
                                           const int *ent_vslot = nullptr) {
  using TR = DT<T, D, G, NW, NST>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tq = lane >> 3, dg = lane & 7;
  const int stp = a.ps / 16;  // tiles per page
  const int ntiles = n_ent * stp;
  unsigned char *my_stages = stages + (size_t)warp * NST * TR::STAGE;
  float2 *pp = pp_all + warp * 16 * G;
  const int cw0 = cw;
  auto tile_rows = [&](int it) -> int {
    const int e = stp == 1 ? it : it / stp, sub = it - e * stp;
    return min(16, ent_valid[e] - sub * 16);
  };
  // lane 0 issues the K and V tile copies of the warp's k-th tile; a tile without rows still
  // arrives (0 bytes) so every stage's phases stay in step.
  auto issue = [&](int k) {
    const int it = warp + k * NW;
    if (it >= ntiles) return;
    if (lane == 0) {
      const int stg = (cw0 + k) % NST;
      const uint32_t bar = smem_u32(&bars[warp][stg]);
      const int e = stp == 1 ? it : it / stp, sub = it - e * stp;
      const int nv = min(16, ent_valid[e] - sub * 16);
      if (nv > 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, (kHostV ? 1u : 2u) * TR::TILE);
        const uint32_t sK = smem_u32(my_stages + (size_t)stg * TR::STAGE);
        const int row = ent_blk[e] * a.ps + sub * 16;
        const uint64_t pol = l2_evict_first_policy();  // K/V rows are read once per step
        tma_load_3d_stream(sK, tmK, 0, h >> a.kv_shift, row, bar, pol);  // the unit head's cache head
        if (!kHostV) tma_load_3d_stream(sK + TR::TILE, tmV, 0, h >> a.kv_shift, row, bar, pol);
      } else {
        mbar_arrive_expect_tx(bar, 0u);
      }
    }
  };

#pragma unroll
  for (int k = 0; k < NST - 1; ++k) issue(k);
  if (q_seq >= 0) load_q<T, D, G, NW, NST>(a, q_seq, h, dg, q2);
  int k = 0;
  static_assert(!kHostV || TR::VPL * TR::ES == 8, "the host value path loads 8 bytes per lane and row");
  for (int cur = warp; cur < ntiles; ++k, cur += NW) {
    issue(k + NST - 1);
    uint2 vh[kHostV ? 16 : 1];  // kHostV: this lane's V slice of the tile's rows
    if constexpr (kHostV) host_v_rows<T, D>(a, h, cur, ntiles, NW, stp, ent_blk, ent_valid, ent_vslot, vh);
    const int stage = (cw0 + k) % NST;
    mbar_wait(smem_u32(&bars[warp][stage]), ((cw0 + k) / NST) & 1, a.ws);
    const int nv = tile_rows(cur);
    if (nv > 0) {
      const unsigned char *sK = my_stages + (size_t)stage * TR::STAGE;  // landed: waited above
      const unsigned char *sV = sK + TR::TILE;
      // ---- QK ----
      float v[TR::NV];
      {
        float2 acc[4][G];
#pragma unroll
        for (int tt = 0; tt < 4; ++tt)
#pragma unroll
          for (int g = 0; g < G; ++g) acc[tt][g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          const unsigned char *rowp = sK + (tt * 4 + tq) * TR::ROW;
#pragma unroll
          for (int c = 0; c < TR::CPL; ++c) {
            const uint4 kw = *reinterpret_cast<const uint4 *>(rowp + (dg + 8 * c) * 16);
            float2 kf[TR::EPC / 2];
            Elem<T>::to_f2(kw, kf);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int e = 0; e < TR::EPC / 2; ++e)
                acc[tt][g] = ffma2(q2[g][c * TR::EPC / 2 + e], kf[e], acc[tt][g]);
          }
        }
#pragma unroll
        for (int tt = 0; tt < 4; ++tt)
#pragma unroll
          for (int g = 0; g < G; ++g) v[tt * G + g] = acc[tt][g].x + acc[tt][g].y;
      }
      reduce_dg<TR::NV>(v, lane);
      // lane holds token t for heads hb * KEEP + j (G >= 2), or head 0 (G == 1)
      const int t = (dg >> 1) * 4 + tq;
      const int hb = (G >= 2) ? (dg & 1) : 0;
#pragma unroll
      for (int j = 0; j < TR::KEEP; ++j)
        if (t >= nv) v[j] = -INFINITY;
      float mx[TR::KEEP], oth[TR::KEEP];
#pragma unroll
      for (int j = 0; j < TR::KEEP; ++j) {
        float x = v[j];
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
        mx[j] = x;
        oth[j] = (G >= 2) ? __shfl_xor_sync(0xffffffffu, x, 1) : x;
      }
      float mnew[G];
      bool moved = false;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int j = g % TR::KEEP, half = g / TR::KEEP;
        const float tmax = (G == 1 || half == hb) ? mx[j] : oth[j];
        mnew[g] = fmaxf(m[g], tmax);
        moved |= mnew[g] != m[g];
      }
      if (moved) {  // warp-uniform
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float al = exp2f(m[g] - mnew[g]);
          m[g] = mnew[g];
          l[g] *= al;
          const float2 aa = make_float2(al, al);
#pragma unroll
          for (int e = 0; e < TR::VPL / 2; ++e) O[g][e] = ffma2(O[g][e], aa, make_float2(0.f, 0.f));
        }
      }
      const bool writer = (G >= 2) || ((dg & 1) == 0);
#pragma unroll
      for (int j = 0; j < TR::KEEP; ++j) {
        const int gj = hb * TR::KEEP + j;
        float mg = m[0];
#pragma unroll
        for (int g = 1; g < G; ++g)
          if (g == gj) mg = m[g];
        const float p = exp2f(v[j] - mg);
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g == gj && writer) l[g] += p;
        if (writer) pp[t * G + gj] = make_float2(p, p);
      }
      __syncwarp();
      // ---- PV ----
      auto pv_row = [&](int tk) {
        float2 vf[TR::VPL / 2];
        const unsigned char *vr = sV + tk * TR::ROW + lane * TR::VPL * TR::ES;
        if constexpr (kHostV) {
          Elem<T>::to_f2_8(vh[tk], vf);
        } else if constexpr (TR::VPL * TR::ES == 16) {
          Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(vr), vf);
        } else {
          Elem<T>::to_f2_8(*reinterpret_cast<const uint2 *>(vr), vf);
        }
        const float2 *pr = pp + tk * G;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 pg = pr[g];
#pragma unroll
          for (int e = 0; e < TR::VPL / 2; ++e) O[g][e] = ffma2(pg, vf[e], O[g][e]);
        }
      };
      if (nv == 16) {
#pragma unroll
        for (int tk = 0; tk < 16; ++tk) pv_row(tk);
      } else if constexpr (kHostV) {  // unrolled, so that vh stays in registers
#pragma unroll
        for (int tk = 0; tk < 16; ++tk)
          if (tk < nv) pv_row(tk);
      } else {
        for (int tk = 0; tk < nv; ++tk) pv_row(tk);
      }
    }
    __syncwarp();
  }
  cw = cw0 + k;
}

// ---- tensor-core tiles (bf16) -------------------------------------------------------------------
// Warp state of warp_tiles_mma. In the m16n8k16 fragments row g = lane / 4 is query head g
// (rows G .. 7 are zero padding of q) and lane % 4 = t4 picks the columns 2 t4, 2 t4 + 1 of each
// 8-column block. O rows g hold P_hi V and rows 8 + g hold P_lo V (see warp_tiles_mma).
template <int D, int G>
struct MmaWarp {
  static_assert(G >= 1 && G <= 8, "query heads are the MMA rows 0..7");
  static constexpr int KS = D / 16;  // k-steps of q K^T
  static constexpr int NT = D / 8;   // 8-column blocks of O
  uint32_t qa[KS][2];  // q as the A operand: a0 (columns 2 t4, + 1) and a2 (+ 8) of each k-step
  float m, l;          // row g: running max of the log2-domain logits, this lane's share of the sum
  float O[NT][4];      // O[n] = {row g: cols 8n + 2t4, +1; row 8 + g: the same cols}
  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;
  }
  __device__ __forceinline__ void load_q(const DecodeArgs &a, int i, int h) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    if (g < G) {
      const uint32_t *qr = reinterpret_cast<const uint32_t *>(reinterpret_cast<const bf16_t *>(a.q) +
                                                              ((size_t)i * a.H_q + (size_t)h * G + g) * D);
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        qa[s][0] = __ldg(qr + 8 * s + t4);
        qa[s][1] = __ldg(qr + 8 * s + 4 + t4);
      }
    } else {
#pragma unroll
      for (int s = 0; s < KS; ++s) qa[s][0] = qa[s][1] = 0u;
    }
  }
  // (m, l, O) of the warp into the CTA merge's shared arrays (see cta_partial).
  __device__ __forceinline__ void stash(float *wO, float *wML) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t4 = lane & 3;
    float lt = l + __shfl_xor_sync(0xffffffffu, l, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    if (g < G) {
      float *o = wO + (size_t)(warp * G + g) * D + 2 * t4;
#pragma unroll
      for (int n = 0; n < NT; ++n)
        *reinterpret_cast<float2 *>(o + 8 * n) = make_float2(O[n][0] + O[n][2], O[n][1] + O[n][3]);
      if (t4 == 0) {
        wML[(warp * G + g) * 2] = m;
        wML[(warp * G + g) * 2 + 1] = lt;
      }
    }
  }
};

// warp_tiles on the tensor cores (bf16): the same tile walk and TMA ring, with each K and V tile
// fetched as D / 64 boxes of 64 elements x 16 rows (128-byte swizzle: chunk c of row t at
// ((c ^ (t % 8)) * 16) inside its 128-byte row). Per 16-token tile:
//   S[g][t]  = sum_d q[g][d] K[t][d]: D/16 k-steps, each one ldmatrix (K rows as the column-major
//              B operand of two 8-token blocks) and two MMAs;
//   online softmax on the lane's four logits (tokens 2 t4, 2 t4 + 1, 8 + 2 t4, 9 + 2 t4), row max
//              by two shuffles, rescale only when some row's max moved;
//   P = exp2(x - m): A rows g = bf16(P), rows 8 + g = bf16(P - bf16(P)) (exact residual);
//   O += P V:  D/16 transposed ldmatrix of V and D/8 MMAs.
// V rows past the live tokens are zeroed first (P is 0 there, but 0 * NaN is NaN); K rows there
// only reach their own logits, which are masked to -inf.
// kHostV: V rows from the value tier (host_v_rows) into registers, then into the tile's V stage
// in the same swizzled layout, so the arithmetic is the same as with V in HBM.
template <int D, int G, int NW, int NST, bool kHostV = false>
__device__ __forceinline__ void warp_tiles_mma(const DecodeArgs &a, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                               int h, int q_seq, MmaWarp<D, G> &w, const int *ent_blk,
                                               const int *ent_valid, int n_ent, unsigned char *stages,
                                               uint64_t (*bars)[NST], int &cw, const int *ent_vslot = nullptr) {
  using TR = DT<bf16_t, D, G, NW, NST>;
  static_assert(TR::ROW % 128 == 0 && TR::TILE % 1024 == 0, "rows of whole 128-byte boxes");
  constexpr int NB = TR::ROW / 128;  // boxes per row
  constexpr int BOX = 16 * 128;      // bytes of one box (16 rows)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int stp = a.ps / 16;  // tiles per page
  const int ntiles = n_ent * stp;
  unsigned char *my_stages = stages + (size_t)warp * NST * TR::STAGE;
  const int cw0 = cw;
  auto issue = [&](int k) {
    const int it = warp + k * NW;
    if (it >= ntiles) return;
    if (lane == 0) {
      const int stg = (cw0 + k) % NST;
      const uint32_t bar = smem_u32(&bars[warp][stg]);
      const int e = stp == 1 ? it : it / stp, sub = it - e * stp;
      const int nv = min(16, ent_valid[e] - sub * 16);
      if (nv > 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, (kHostV ? 1u : 2u) * TR::TILE);
        const uint32_t sK = smem_u32(my_stages + (size_t)stg * TR::STAGE);
        const int row = ent_blk[e] * a.ps + sub * 16;
        const uint64_t pol = l2_evict_first_policy();  // K/V rows are read once per step
#pragma unroll
        for (int b = 0; b < NB; ++b) {  // x = 64 b elements: 128-byte aligned
          tma_load_3d_stream(sK + b * BOX, tmK, b * 64, h >> a.kv_shift, row, bar, pol);
          if (!kHostV) tma_load_3d_stream(sK + TR::TILE + b * BOX, tmV, b * 64, h >> a.kv_shift, row, bar, pol);
        }
      } else {
        mbar_arrive_expect_tx(bar, 0u);
      }
    }
  };

#pragma unroll
  for (int k = 0; k < NST - 1; ++k) issue(k);
  if (q_seq >= 0) w.load_q(a, q_seq, h);
  const float qs = a.scale * kLog2e;
  const int t4 = lane & 3, r8 = lane & 7, mi = lane >> 3;
  // ldmatrix row of this lane: K matrix mi = (token block mi / 2, chunk 2s + mi % 2); V matrix
  // mi = (token block mi % 2, chunk 2n + mi / 2); the row is the token, so (row % 8) = r8
  const uint32_t k_row = (uint32_t)(((mi >> 1) * 8 + r8) * 128);
  const int k_ch = mi & 1;
  const uint32_t v_row = (uint32_t)(((mi & 1) * 8 + r8) * 128);
  const int v_ch = mi >> 1;
  int k = 0;
  for (int cur = warp; cur < ntiles; ++k, cur += NW) {
    issue(k + NST - 1);
    uint2 vh[kHostV ? 16 : 1];
    if constexpr (kHostV) host_v_rows<bf16_t, D>(a, h, cur, ntiles, NW, stp, ent_blk, ent_valid, ent_vslot, vh);
    const int stage = (cw0 + k) % NST;
    mbar_wait(smem_u32(&bars[warp][stage]), ((cw0 + k) / NST) & 1, a.ws);
    const int e = stp == 1 ? cur : cur / stp, sub = cur - e * stp;
    const int nv = min(16, ent_valid[e] - sub * 16);
    if (nv > 0) {
      unsigned char *sV = my_stages + (size_t)stage * TR::STAGE + TR::TILE;
      if constexpr (kHostV) {
        // lane's 8 bytes of row t: chunk lane / 2 of the row, half lane % 2 (rows past nv are zero)
        const int ch = lane >> 1;
#pragma unroll
        for (int t = 0; t < 16; ++t)
          *reinterpret_cast<uint2 *>(sV + (ch >> 3) * BOX + t * 128 + (((ch & 7) ^ (t & 7)) << 4) + (lane & 1) * 8) =
              vh[t];
      }
      const uint32_t aK = smem_u32(my_stages + (size_t)stage * TR::STAGE), aV = smem_u32(sV);
      // ---- S = q K^T ----
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < MmaWarp<D, G>::KS; ++s) {
        const int ch = 2 * s + k_ch;
        uint32_t kb[4];
        ldsm_x4(aK + (ch >> 3) * BOX + k_row + (((ch & 7) ^ r8) << 4), kb);
        const uint32_t qa4[4] = {w.qa[s][0], 0u, w.qa[s][1], 0u};
        mma_16816_bf16(s0, qa4, kb[0], kb[1]);
        mma_16816_bf16(s1, qa4, kb[2], kb[3]);
      }
      // ---- online softmax, row g ----
      const int tb = 2 * t4;
      float x[4] = {s0[0] * qs, s0[1] * qs, s1[0] * qs, s1[1] * qs};
      if (tb >= nv) x[0] = -INFINITY;
      if (tb + 1 >= nv) x[1] = -INFINITY;
      if (tb + 8 >= nv) x[2] = -INFINITY;
      if (tb + 9 >= nv) x[3] = -INFINITY;
      float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float mnew = fmaxf(w.m, tmax);  // finite: token 0 of a tile is always live
      if (__any_sync(0xffffffffu, mnew != w.m)) {
        const float al = exp2f(w.m - mnew);  // 0 when m was -inf, 1 when it did not move
        w.m = mnew;
        w.l *= al;
#pragma unroll
        for (int n = 0; n < MmaWarp<D, G>::NT; ++n)
#pragma unroll
          for (int j = 0; j < 4; ++j) w.O[n][j] *= al;
      }
      float p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = exp2f(x[j] - w.m);
      w.l += (p[0] + p[1]) + (p[2] + p[3]);
      uint32_t pa[4];
      pa[0] = pack_bf16x2(p[0], p[1]);
      pa[2] = pack_bf16x2(p[2], p[3]);
      pa[1] = pack_bf16x2(p[0] - bf16_lo(pa[0]), p[1] - bf16_hi(pa[0]));
      pa[3] = pack_bf16x2(p[2] - bf16_lo(pa[2]), p[3] - bf16_hi(pa[2]));
      // ---- O += P V ----
      if (!kHostV && nv < 16) {  // whole rows, so the swizzle does not matter
        for (int z = lane; z < (16 - nv) * (D / 8); z += 32) {
          const int t = nv + z / (D / 8), ch = z % (D / 8);
          *reinterpret_cast<uint4 *>(sV + (ch >> 3) * BOX + t * 128 + (ch & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();  // V rows written by the warp (zeros, or the value tier's rows) before ldmatrix
#pragma unroll
      for (int n2 = 0; n2 < D / 16; ++n2) {
        const int ch = 2 * n2 + v_ch;
        uint32_t vb[4];
        ldsm_x4_trans(aV + (ch >> 3) * BOX + v_row + (((ch & 7) ^ r8) << 4), vb);
        mma_16816_bf16(w.O[2 * n2], pa, vb[0], vb[1]);
        mma_16816_bf16(w.O[2 * n2 + 1], pa, vb[2], vb[3]);
      }
    }
    __syncwarp();
  }
  cw = cw0 + k;
}

// The CTA merge of its warps' states, stashed in shared memory by the warps (per warp w and head
// g: O row wO[(w G + g) D ..] relative to m, and (m, l) at wML[(w G + g) 2]); the caller has
// synchronised after the stash. cta_partial writes one partial (m, l and O relative to m) at
// `slot`; cta_output writes the G output rows normalised by l (a unit one CTA covers entirely).
template <int D, int G, int NW>
__device__ __forceinline__ float cta_merge_elem(const float *wO, const float *wML, int g, int d, float *M_out,
                                                float *L_out) {
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, wML[(w * G + g) * 2]);
  float acc = 0.f, L = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sc = exp2f(wML[(w * G + g) * 2] - M);
      acc = fmaf(sc, wO[(w * G + g) * D + d], acc);
      L = fmaf(sc, wML[(w * G + g) * 2 + 1], L);
    }
  }
  *M_out = M;
  *L_out = L;
  return acc;
}
template <int D, int G, int NW>
__device__ __forceinline__ void cta_partial(const DecodeArgs &a, size_t slot, const float *wO, const float *wML) {
  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float M, L;
    a.part_o[(slot * G + g) * D + d] = cta_merge_elem<D, G, NW>(wO, wML, g, d, &M, &L);
    if (d == 0) {
      a.part_ml[(slot * G + g) * 2] = M;
      a.part_ml[(slot * G + g) * 2 + 1] = L;
    }
  }
}
template <typename T, int D, int G, int NW>
__device__ __forceinline__ void cta_output(const DecodeArgs &a, int unit, const float *wO, const float *wML) {
  T *out = reinterpret_cast<T *>(a.out) + ((size_t)(unit / a.H_kv) * a.H_q + (size_t)(unit % a.H_kv) * G) * D;
  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float M, L;
    const float acc = cta_merge_elem<D, G, NW>(wO, wML, g, d, &M, &L);
    Elem<T>::store(out + idx, L > 0.f ? acc / L : 0.f);
  }
}

// The FMA warp state (O over dims lane * VPL .., l a per-lane share) into the merge's arrays.
template <typename T, int D, int G, int NW, int NST>
__device__ __forceinline__ void stash_fma(float (&m)[G], float (&l)[G], float2 (&O)[G][DT<T, D, G, NW, NST>::VPL / 2],
                                          float *wO, float *wML) {
  using TR = DT<T, D, G, NW, NST>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float x = l[g];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
#pragma unroll
    for (int e = 0; e < TR::VPL / 2; ++e)
      reinterpret_cast<float2 *>(wO + (warp * G + g) * D + lane * TR::VPL)[e] = O[g][e];
    if (lane == 0) {
      wML[(warp * G + g) * 2] = m[g];
      wML[(warp * G + g) * 2 + 1] = x;
    }
  }
}

template <typename T, int D, int G, int NW, int NST>
struct DecodeSmem {
  using TR = DT<T, D, G, NW, NST>;
  unsigned char *stages;
  float2 *pp_all;
  float *wML;
  int *ent_blk, *ent_valid, *ent_vslot;
  int *extra;  // flat layout: the unit prefix sums
  __device__ explicit DecodeSmem(unsigned char *raw) {
    stages = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    pp_all = reinterpret_cast<float2 *>(stages + TR::STAGES);
    wML = reinterpret_cast<float *>(pp_all + NW * 16 * G);
    ent_blk = reinterpret_cast<int *>(wML + NW * G * 2);
    ent_valid = ent_blk + kSwMax;
    ent_vslot = ent_valid + kSwMax;
    extra = ent_vslot + kSwMax;
  }
};

// ---- split layout: one CTA per (split of `sw` list entries, KV head, sequence) ----------------
// kMma: the tensor-core tiles (bf16, V in HBM; the tensor maps are the swizzled 128-byte boxes).
template <typename T, int D, int G, int NW, int NST, bool kHostV, bool kMma = false>
__global__ void __launch_bounds__(NW * 32) decode_split_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV) {
  static_assert(!kMma || sizeof(T) == 2, "tensor-core tiles: bf16");
  pdl_wait();  // dependents are released when this grid completes
  using TR = DT<T, D, G, NW, NST>;
  extern __shared__ __align__(128) unsigned char smem_dyn[];
  DecodeSmem<T, D, G, NW, NST> sm(smem_dyn);
  __shared__ __align__(8) uint64_t bars[NW][NST];
  __shared__ int flag_last;

  // blockIdx.x = unit, blockIdx.y = split: CTAs are launched split-major, so every unit's first
  // (full) splits run before the shorter last splits and the tail of the grid is short work
  const int unit = blockIdx.x, s = blockIdx.y;
  const int i = unit / a.H_kv, h = unit - i * a.H_kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  const int e0 = split_off(s, a.sw, a.taper), len = split_len(s, a.sw, a.taper);
  const size_t pbase = (size_t)unit * a.n_items_max + s;

  // the list entry the alone test below reads, issued with the others (independent of them)
  const int32_t sw_entry =
      (a.selected && a.n_items_max > 1 && a.b_max > a.sw) ? a.selected[(size_t)unit * a.b_max + a.sw] : -1;
  int n_ent = 0;
  if (seq_len < 1 || P > a.max_pages) {
    if (s == 0 && tid == 0) set_status(a.ws, PSK_DEV_BAD_SEQLEN);
  } else if (a.selected) {
    const int32_t *row = a.selected + (size_t)unit * a.b_max;
    if (e0 < a.b_max && row[e0] >= 0) n_ent = min(len, a.b_max - e0);
  } else if (e0 < P) {
    n_ent = min(len, P - e0);
  }
  if (lane == 0) {
    for (int k = 0; k < NST; ++k) mbar_init(smem_u32(&bars[warp][k]), 1);
    fence_mbar_init();
  }
  load_entries<NW * 32>(a, i, unit, P, seq_len, e0, n_ent, sm.ent_blk, sm.ent_valid, kHostV ? sm.ent_vslot : nullptr);
  __syncthreads();

  // a unit whose whole list fits this split (sparse: no entry at index sw) needs no partials and
  // no merge: split 0 writes the normalised output and the other splits leave at once
  bool alone = false;
  if (a.selected) {
    alone = a.n_items_max == 1 || a.b_max <= a.sw || sw_entry < 0;
  } else {
    alone = a.n_items_max == 1 || P <= a.sw;
  }
  if (alone && s > 0) return;

  if (n_ent > 0) {
    float *wO = reinterpret_cast<float *>(sm.stages);  // the merge reuses the stages
    int cw = 0;
    if constexpr (kMma) {
      MmaWarp<D, G> w;
      w.reset();
      warp_tiles_mma<D, G, NW, NST, kHostV>(a, &tmK, &tmV, h, i, w, sm.ent_blk, sm.ent_valid, n_ent, sm.stages, bars,
                                            cw, kHostV ? sm.ent_vslot : nullptr);
      __syncthreads();  // every warp is done with the stages
      w.stash(wO, sm.wML);
    } else {
      float2 q2[G][TR::CPL * TR::EPC / 2];  // loaded by warp_tiles, behind the first tile copies
      float m[G], l[G];
      float2 O[G][TR::VPL / 2];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < TR::VPL / 2; ++e) O[g][e] = make_float2(0.f, 0.f);
      }
      warp_tiles<T, D, G, NW, NST, kHostV>(a, &tmK, &tmV, h, i, q2, sm.ent_blk, sm.ent_valid, n_ent, sm.stages,
                                           sm.pp_all, bars, cw, m, l, O, kHostV ? sm.ent_vslot : nullptr);
      __syncthreads();  // every warp is done with the stages
      stash_fma<T, D, G, NW, NST>(m, l, O, wO, sm.wML);
    }
    __syncthreads();
    if (alone) {
      cta_output<T, D, G, NW>(a, unit, wO, sm.wML);
      return;
    }
    cta_partial<D, G, NW>(a, pbase, wO, sm.wML);
  } else if (alone) {  // nothing to read and nothing to merge: zero rows
    T *out = reinterpret_cast<T *>(a.out) + ((size_t)i * a.H_q + (size_t)h * G) * D;
    for (int idx = tid; idx < G * D; idx += NW * 32) Elem<T>::store(out + idx, 0.f);
    return;
  } else if (tid < G) {  // nothing to read: an empty partial
    a.part_ml[(pbase * G + tid) * 2] = -INFINITY;
    a.part_ml[(pbase * G + tid) * 2 + 1] = 0.f;
  }

  // ---- the last CTA of the unit merges the partials ------------------------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(a.tickets + unit, 1u);
    flag_last = prev == (unsigned)(a.n_items_max - 1);
  }
  __syncthreads();
  if (!flag_last) return;
  __threadfence();
  if (tid == 0) a.tickets[unit] = 0u;
  merge_unit<T, D, G, NW, true>(a, unit, (size_t)unit * a.n_items_max, a.n_items_max, reinterpret_cast<float *>(sm.stages),
                          sm.wML);
}

// ---- flat layout ---------------------------------------------------------------------------------
// List entries per unit of a sparse call: one past the last non-negative id of the unit's row
// (0 for a sequence whose length is out of range). One warp per unit.
__global__ void decode_counts_kernel(DecodeArgs a) {
  pdl_begin();
  const int unit = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (unit >= a.B * a.H_kv) return;
  const int i = unit / a.H_kv;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  int last = -1;
  if (seq_len >= 1 && P <= a.max_pages) {
    const int32_t *row = a.selected + (size_t)unit * a.b_max;
    for (int x = lane; x < a.b_max; x += 32)
      if (row[x] >= 0) last = x;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0) a.counts[unit] = last + 1;
}

// A persistent grid of C CTAs cuts the concatenation of all units' lists (E entries) into C
// equal shares: CTA c streams entries [c E / C, (c + 1) E / C), which may cover the end of one
// unit, whole units and the start of another. Each (CTA, unit) segment leaves one partial at
// slot c + u (unique: shares are ordered like the units), and the last CTA of a unit to finish
// (ticket, no waiting) merges the unit's partials. Units without entries get zero rows from CTA
// u % C. Balancing by entries removes the tail that budget-sized splits leave when budgets differ.
template <typename T, int D, int G, int NW, int NST, bool kMma = false>
__global__ void __launch_bounds__(NW * 32) decode_flat_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                                                              const __grid_constant__ CUtensorMap tmV) {
  static_assert(!kMma || sizeof(T) == 2, "tensor-core tiles: bf16");
  pdl_wait();  // dependents are released when this grid completes
  using TR = DT<T, D, G, NW, NST>;
  constexpr int NT = NW * 32;
  extern __shared__ __align__(128) unsigned char smem_dyn[];
  DecodeSmem<T, D, G, NW, NST> sm(smem_dyn);
  int *start = sm.extra;  // [U + 1] exclusive prefix of the units' entry counts
  __shared__ __align__(8) uint64_t bars[NW][NST];
  __shared__ int flag_last;
  __shared__ int scan_tot[NW];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int U = a.B * a.H_kv;
  const int c = blockIdx.x;

  // ---- entry counts and their prefix sums ----------------------------------------------------
  for (int u = tid; u < U; u += NT) {  // coalesced, independent loads
    int cnt;
    if (a.selected) {
      cnt = a.counts[u];
    } else {
      const int sl = a.seq_lens[u / a.H_kv];
      const int P = (sl + a.ps - 1) / a.ps;
      cnt = (sl >= 1 && P <= a.max_pages) ? P : 0;
    }
    start[u + 1] = cnt;
  }
  __syncthreads();
  const int per = (U + NT - 1) / NT;  // contiguous units per thread for the scan
  const int u0 = min(U, tid * per), u1 = min(U, u0 + per);
  int run = 0;
  for (int u = u0; u < u1; ++u) run += start[u + 1];
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scan_tot[warp] = incl;
  if (lane == 0) {
    for (int k = 0; k < NST; ++k) mbar_init(smem_u32(&bars[warp][k]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  int base = incl - run;
  for (int w = 0; w < warp; ++w) base += scan_tot[w];
  for (int u = u0; u < u1; ++u) {
    const int cnt = start[u + 1];
    start[u + 1] = base + cnt;
    base += cnt;
  }
  if (tid == 0) start[0] = 0;
  __syncthreads();
  const long long E = start[U];
  // CTAs with a share: every share holds at least kFlatMinShare entries (and is never empty)
  const int C = (int)min((long long)gridDim.x, max(1LL, E / kFlatMinShare));

  // ---- units without entries: zero rows (and the status for a bad length) ----------------------
  for (int u = c; u < U; u += gridDim.x) {
    if (start[u + 1] != start[u]) continue;
    const int i = u / a.H_kv;
    const int sl = a.seq_lens[i];
    if ((sl < 1 || (sl + a.ps - 1) / a.ps > a.max_pages) && (u % a.H_kv) == 0 && tid == 0)
      set_status(a.ws, PSK_DEV_BAD_SEQLEN);
    T *out = reinterpret_cast<T *>(a.out) + ((size_t)i * a.H_q + (size_t)(u % a.H_kv) * G) * D;
    for (int idx = tid; idx < G * D; idx += NT) Elem<T>::store(out + idx, 0.f);
  }
  if (c >= C) return;

  auto cta_of = [&](long long e) -> int {  // the CTA whose share holds entry e
    return (int)min((long long)C - 1, ((e + 1) * C - 1) / E);
  };
  const long long e_lo = (long long)c * E / C, e_hi = (long long)(c + 1) * E / C;
  int u;
  {  // the unit holding entry e_lo: the last u with start[u] <= e_lo
    int lo = 0, hi = U - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start[mid] <= e_lo) lo = mid; else hi = mid - 1;
    }
    u = lo;
  }
  int cw = 0;
  for (long long e = e_lo; e < e_hi;) {
    while (start[u + 1] <= e) ++u;  // skip units without entries
    const long long seg_end = min(e_hi, (long long)start[u + 1]);
    const int i = u / a.H_kv, h = u % a.H_kv;
    const int seq_len = a.seq_lens[i];
    const int P = (seq_len + a.ps - 1) / a.ps;
    float *wO = reinterpret_cast<float *>(sm.stages);  // the merge reuses the stages
    if constexpr (kMma) {
      MmaWarp<D, G> w;
      w.reset();
      w.load_q(a, i, h);
      for (long long x0 = e; x0 < seg_end; x0 += kSwMax) {
        const int n = (int)min((long long)kSwMax, seg_end - x0);
        __syncthreads();  // the previous entry table and stages are no longer in use
        load_entries<NT>(a, i, u, P, seq_len, (int)(x0 - start[u]), n, sm.ent_blk, sm.ent_valid);
        __syncthreads();
        warp_tiles_mma<D, G, NW, NST>(a, &tmK, &tmV, h, -1, w, sm.ent_blk, sm.ent_valid, n, sm.stages, bars, cw);
      }
      __syncthreads();  // every warp is done with the stages
      w.stash(wO, sm.wML);
    } else {
      float2 q2[G][TR::CPL * TR::EPC / 2];
      load_q<T, D, G, NW, NST>(a, i, h, lane & 7, q2);
      float m[G], l[G];
      float2 O[G][TR::VPL / 2];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int x = 0; x < TR::VPL / 2; ++x) O[g][x] = make_float2(0.f, 0.f);
      }
      for (long long x0 = e; x0 < seg_end; x0 += kSwMax) {
        const int n = (int)min((long long)kSwMax, seg_end - x0);
        __syncthreads();  // the previous entry table and stages are no longer in use
        load_entries<NT>(a, i, u, P, seq_len, (int)(x0 - start[u]), n, sm.ent_blk, sm.ent_valid);
        __syncthreads();
        warp_tiles<T, D, G, NW, NST>(a, &tmK, &tmV, h, -1, q2, sm.ent_blk, sm.ent_valid, n, sm.stages, sm.pp_all, bars,
                                     cw, m, l, O);
      }
      __syncthreads();  // every warp is done with the stages
      stash_fma<T, D, G, NW, NST>(m, l, O, wO, sm.wML);
    }
    __syncthreads();
    cta_partial<D, G, NW>(a, (size_t)c + u, wO, sm.wML);
    const int c_first = cta_of(start[u]), c_last = cta_of((long long)start[u + 1] - 1);
    const int nseg = c_last - c_first + 1;
    __threadfence();
    __syncthreads();
    if (tid == 0) flag_last = atomicAdd(a.tickets + u, 1u) == (unsigned)(nseg - 1);
    __syncthreads();
    if (flag_last) {
      __threadfence();
      if (tid == 0) a.tickets[u] = 0u;
      merge_unit<T, D, G, NW, false>(a, u, (size_t)c_first + u, nseg, reinterpret_cast<float *>(sm.stages), sm.wML);
    }
    e = seg_end;
  }
}

// Value tier fill: entry x = (sequence, cache head, page, slot). slot >= 0 copies the page's
// ps rows of that head from the host value cache (over NVLink-C2C) into hot-buffer slot `slot`
// and records it in v_slot; slot < 0 clears the page's record (its V is read from the host
// again). One CTA per entry, 16 bytes per thread and step.
__global__ void value_tier_fill_kernel(const uint16_t *v_host, const int32_t *block_table, const int32_t *entries,
                                       uint16_t *v_hot, int32_t *v_slot, void *ws, int H_kv, int D, int ps, int nb,
                                       int max_pages, int B, int n_slots) {
  pdl_begin();
  const int32_t *ent = entries + (size_t)blockIdx.x * 4;
  const int i = ent[0], h = ent[1], p = ent[2], slot = ent[3];
  if (i < 0 || i >= B || h < 0 || h >= H_kv || p < 0 || p >= max_pages || slot >= n_slots) {
    if (threadIdx.x == 0) set_status(ws, PSK_DEV_BAD_SELECTED);
    return;
  }
  int32_t *rec = v_slot + ((size_t)i * H_kv + h) * max_pages + p;
  if (slot < 0) {
    if (threadIdx.x == 0) *rec = -1;
    return;
  }
  const int blk = block_table[(size_t)i * max_pages + p];
  if (blk < 0 || blk >= nb) {
    if (threadIdx.x == 0) set_status(ws, PSK_DEV_BAD_BLOCK);
    return;
  }
  const int cpr = D / 8;  // 16-byte chunks per row
  for (int x = threadIdx.x; x < ps * cpr; x += blockDim.x) {
    const int r = x / cpr, c = x - r * cpr;
    const uint4 v = *reinterpret_cast<const uint4 *>(v_host + (((size_t)blk * ps + r) * H_kv + h) * D + c * 8);
    *reinterpret_cast<uint4 *>(v_hot + ((size_t)slot * ps + r) * D + c * 8) = v;
  }
  if (threadIdx.x == 0) *rec = slot;
}

// G = 8 is built on the tensor cores only (the FMA tiles' per-lane q would not fit).
template <typename T, int D, int G>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t s) {
  constexpr int NW = 4, NST = 2;
  using TR = DT<T, D, G, NW, NST>;
  static_assert(TR::STAGES >= (size_t)kMaxItems * G * 4, "stage memory must hold the merge weights");
  static_assert(TR::STAGES >= (size_t)kFlatMaxCtas * G * 4, "stage memory must hold the merge weights");
  // bf16: the tensor-core tiles (unless PSK_DECODE_MMA=0)
  constexpr bool kMmaOk = sizeof(T) == 2 && D % 64 == 0;
  constexpr bool kFmaOk = G <= 4;
  const bool mma = kMmaOk && (tuning().decode_mma || !kFmaOk);
  if (!mma && !kFmaOk) return cudaErrorInvalidValue;
  CUtensorMap tmK, tmV;
  const long long rows = (long long)a.nb * a.ps;
  const int dt = sizeof(T) == 4 ? PSK_F32 : PSK_BF16;
  // host values: no tensor map over host memory (V is read with plain loads); tmV repeats tmK
  if (!encode_cache_map(&tmK, a.k_cache, dt, D, a.H_kv_cache, rows, 16, mma) ||
      !encode_cache_map(&tmV, a.v_host ? a.k_cache : a.v_cache, dt, D, a.H_kv_cache, rows, 16, mma))
    return cudaErrorInvalidValue;
  if (a.v_host) {  // the value tier: sparse split layout only
    if constexpr (sizeof(T) == 2 && D == 128) {
      if (a.flat || !a.selected) return cudaErrorInvalidValue;
      dim3 grid(a.B * a.H_kv, a.n_items_max);
      if (mma) {
        // the same warp layout as the HBM decode below, so the two give identical bits
        if ((long long)grid.x * grid.y < sm_count())
          return launch_kernel(true, decode_split_kernel<T, D, G, 2 * NW, NST, true, true>, grid, 2 * NW * 32,
                               DT<T, D, G, 2 * NW, NST>::SMEM, s, a, tmK, tmV);
        return launch_kernel(true, decode_split_kernel<T, D, G, NW, NST, true, true>, grid, NW * 32, TR::SMEM, s, a, tmK,
                             tmV);
      }
      if constexpr (kFmaOk)
        return launch_kernel(true, decode_split_kernel<T, D, G, NW, NST, true>, grid, NW * 32, TR::SMEM, s, a, tmK,
                             tmV);
    }
    return cudaErrorInvalidValue;
  }
  if (!a.flat) {
    dim3 grid(a.B * a.H_kv, a.n_items_max);
    if constexpr (kMmaOk) {
      if (mma) {
        // A grid smaller than one CTA per SM (small batches): eight warps per CTA, so the
        // split's tiles run side by side instead of two after another per warp (B = 1, 32K
        // context: 33.8 against 35.8 us per step; on the batched workload four warps and three
        // CTAs per SM stay faster, 92 against 125 us)
        if ((long long)grid.x * grid.y < sm_count())
          return launch_kernel(true, decode_split_kernel<T, D, G, 2 * NW, NST, false, true>, grid, 2 * NW * 32,
                               DT<T, D, G, 2 * NW, NST>::SMEM, s, a, tmK, tmV);
        return launch_kernel(true, decode_split_kernel<T, D, G, NW, NST, false, true>, grid, NW * 32, TR::SMEM, s, a,
                             tmK, tmV);
      }
    }
    if constexpr (kFmaOk)
      return launch_kernel(true, decode_split_kernel<T, D, G, NW, NST, false>, grid, NW * 32, TR::SMEM, s, a, tmK,
                           tmV);
    return cudaErrorInvalidValue;
  }
  const int U = a.B * a.H_kv;
  cudaError_t e;
  if (a.selected) {
    e = launch_kernel(true, decode_counts_kernel, (U + 7) / 8, 256, 0, s, a);
    if (e != cudaSuccess) return e;
  }
  const size_t smem = TR::SMEM + (size_t)(U + 1) * 4;
  auto flat_launch = [&](auto kfn) -> cudaError_t {
    int per_sm = 0;
    cudaError_t e2 = kernel_setup(reinterpret_cast<const void *>(kfn), NW * 32, smem, &per_sm);
    if (e2 != cudaSuccess) return e2;
    const int ctas = std::max(1, std::min(kFlatMaxCtas, sm_count() * std::max(1, per_sm)));
    return launch_kernel(!a.selected, kfn, ctas, NW * 32, smem, s, a, tmK, tmV);
  };
  if constexpr (kMmaOk)
    if (mma) return flat_launch(decode_flat_kernel<T, D, G, NW, NST, true>);
  if constexpr (kFmaOk) return flat_launch(decode_flat_kernel<T, D, G, NW, NST>);
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_value_tier_fill(const psk_layout &L, const void *v_host, const int32_t *block_table,
                                   const int32_t *entries, int n_entries, void *v_hot, int n_slots, int32_t *v_slot,
                                   void *ws, cudaStream_t s) {
  if (n_entries == 0) return cudaSuccess;
  return launch_kernel(true, value_tier_fill_kernel, n_entries, 128, 0, s, reinterpret_cast<const uint16_t *>(v_host),
                       block_table, entries, reinterpret_cast<uint16_t *>(v_hot), v_slot, ws, L.num_kv_heads,
                       L.v_head_dim, L.page_size, L.num_blocks, L.max_pages, L.batch, n_slots);
}

bool plan_decode(const psk_layout &L, int entries, bool dense, DecodePlan *plan) {
  const long long units = (long long)L.batch * L.num_kv_heads;
  const int G = L.num_q_heads / L.num_kv_heads;
  // Dense: the flat layout (equal shares of all units' page lists over a persistent grid)
  // whenever its prefix sums fit in shared memory. Sparse: the split layout, measured faster on
  // the batched workload (the flat one adds a count pass over the selected rows and more
  // partials, and short budget lists leave its shares little to balance).
  bool flat = dense && units <= kFlatMaxUnits;
  const Tuning &tu = tuning();
  if (tu.decode_layout == 1) flat = false;                          // tuning override: "split"
  if (tu.decode_layout == 2) flat = units <= kFlatMaxUnits;         // tuning override: "flat"
  size_t slots;
  if (flat) {
    plan->sw = kSwMax;
    plan->n_items_max = 1;
    plan->taper = 0;
    slots = (size_t)kFlatMaxCtas + (size_t)units;
  } else {
    // 64 list entries per CTA (measured best on the batched workload); fewer (down to 8) while
    // the grid would not fill the GPU (all SMs x 2 CTAs) a few times over, more when a unit
    // would need over kMaxItems partials
    int sw = 64;
    const long long fill = 4LL * sm_count() * 2;
    while (sw > 8 && units * ((entries + sw - 1) / sw) < fill) sw /= 2;  // 8: measured best at B = 1
    if (tu.decode_split >= 1 && tu.decode_split <= kSwMax) sw = tu.decode_split;  // tuning override: entries per CTA
    while (sw < kSwMax && (entries + sw - 1) / sw > kMaxItems) sw *= 2;
    plan->sw = sw;
    plan->n_items_max = (entries + sw - 1) / sw;
    plan->taper = 0;
    // sparse lists longer than one split: tapered splits when they stay few enough to merge
    if (!dense && entries > sw && !tu.decode_no_taper) {
      int n = 0;
      while (split_off(n, sw, 1) < entries) ++n;
      if (n <= kMaxItems) {
        plan->taper = 1;
        plan->n_items_max = n;
      }
    }
    slots = (size_t)units * plan->n_items_max;
  }
  plan->flat = flat ? 1 : 0;
  size_t off = ws_scratch_offset((size_t)units);
  plan->off_o = off;
  off = align_up(off + slots * G * L.v_head_dim * 4, 256);
  plan->off_ml = off;
  off = align_up(off + slots * G * 2 * 4, 256);
  plan->off_counts = off;
  off = align_up(off + (size_t)units * 4, 256);
  plan->ws_bytes = off;
  plan->off_tickets = ws_decode_tickets_offset((size_t)units);
  return plan->n_items_max <= kMaxItems;
}

#define PSK_DECODE_CASES(X)   \
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

bool decode_supported(int dtype, int D, int D_v, int G, int ps) {
  if (D_v != D || ps % 16 != 0 || ps > 64) return false;
#define X(TT, DT_, DD, GG) \
  if (dtype == DT_ && D == DD && G == GG) return true;
  PSK_DECODE_CASES(X)
#undef X
  return false;
}

cudaError_t launch_decode(const DecodeArgs &a, int dtype, cudaStream_t s) {
  const int D = a.D, G = a.H_q / a.H_kv;
#define X(TT, DT_, DD, GG) \
  if (dtype == DT_ && D == DD && G == GG) return launch_t<TT, DD, GG>(a, s);
  PSK_DECODE_CASES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace psk
