// Stage 4: exact softmax attention over the selected pages of a GQA paged cache, split-K over
// pages with an fp32 online-softmax (m, l, O) state and a log-sum-exp merge (EntmaxKV README,
// introduction: "the attention is exact over that selection"; LOCKS PKG-INFO, "How it works",
// Sparse decode: a paged kernel that reads only the selected pages). The dense decode is the
// same kernel with the implicit page list 0 .. P-1.
//
// Work: a (sequence, KV head) unit's page list is cut into items of `sw` consecutive list
// entries; items are numbered unit-major. The kernel is persistent: each warp is independent
// and walks items gw, gw + TW, ... (gw = global warp id, TW = warps in the grid). A page is cut
// into 16-token tiles. Every warp runs a producer cursor NST - 1 tiles ahead of its consumer:
// the producer turns the item's list entries into tiles (block-table lookups, bounds checks)
// and issues 16-byte cp.async copies of the K and V rows into a per-warp ring of NST stages
// (rows past seq_len are zero-filled, never read), plus the group's q rows with an item's first
// tile, so the memory pipe stays busy across item boundaries.
//
// Consumer, per tile: lane = (tq = lane / 8, dg = lane % 8). QK: the lane owns the 16-byte
// chunks dg, dg + 8, ... of each K row and the matching q slices (scaled by scale * log2(e) so
// exp2 gives the softmax weights) and computes partial dot products for tokens tq, tq + 4,
// tq + 8, tq + 12 and all G heads of the group with packed fp32x2 FMAs; a transposing
// butterfly over the 8 dg lanes leaves each lane the full logits of one token for G/2 heads.
// Online softmax: tile max per head by 4 shuffles, rescale only when the max moved, p to a
// per-warp array (stored as (p, p) pairs). PV: the lane owns D/32 output dims of all G heads
// and accumulates with packed FMAs from one conflict-free V row chunk per token.
//
// At an item's last tile the warp writes its partial (m, l, O unnormalised) to the workspace
// and takes a ticket for the unit; the warp holding the last ticket (no waiting) merges the
// unit's partials by log-sum-exp and writes the G output rows. Empty items (past the end of
// the list) write an empty partial and take their ticket too.
#include <algorithm>

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSwMax = 256;  // list entries per item, upper bound

template <typename T, int D, int G, int NST>
struct DT {
  static constexpr int ES = Elem<T>::kBytes;
  static constexpr int EPC = Elem<T>::kPerChunk;  // elements per 16-byte chunk
  static constexpr int NC = D / EPC;               // chunks per row
  static constexpr int CPL = NC / 8;               // QK chunks per lane
  static constexpr int VPL = D / 32;               // PV dims per lane
  static constexpr int ROW = D * ES;               // bytes per row
  static constexpr int TILE = 16 * ROW;
  static constexpr int QBYTES = G * ROW;
  static constexpr int STAGE = 2 * TILE + QBYTES;  // K tile, V tile, q rows
  static constexpr int LOADS = 16 * NC / 32;       // 16-byte chunks per lane per tile (each of K, V)
  static constexpr int QCH = G * NC;               // 16-byte chunks of q
  static constexpr int NV = 4 * G;                 // partial logits per lane before reduce
  static constexpr int KEEP = NV >= 8 ? NV / 8 : 1;
  static constexpr size_t SMEM = (size_t)NST * STAGE + 16 * G * 8 + NST * 16 + (size_t)kSwMax * 3 * 4;
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

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ int warp_max_i(int x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ int warp_min_i(int x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = min(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Merge every partial of `unit` (the caller holds the unit's last ticket) into its G output rows.
template <typename T, int D, int G>
__device__ void merge_unit(const DecodeArgs &a, int unit, int lane) {
  constexpr int VPL = D / 32;
  const int i = unit / a.H_kv, h = unit - i * a.H_kv;
  const size_t it0 = (size_t)unit * a.n_items_max;
  float M[G];
#pragma unroll
  for (int g = 0; g < G; ++g) M[g] = -INFINITY;
  for (int s = lane; s < a.n_items_max; s += 32)
#pragma unroll
    for (int g = 0; g < G; ++g) M[g] = fmaxf(M[g], __ldcg(a.part_ml + ((it0 + s) * G + g) * 2));
#pragma unroll
  for (int g = 0; g < G; ++g) M[g] = warp_max(M[g]);
  float L[G], O[G][VPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    L[g] = 0.f;
#pragma unroll
    for (int e = 0; e < VPL; ++e) O[g][e] = 0.f;
  }
#pragma unroll 2
  for (int s = 0; s < a.n_items_max; ++s) {
    const size_t it = it0 + s;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float ms = __ldcg(a.part_ml + (it * G + g) * 2);
      if (ms == -INFINITY) continue;  // empty partial (uniform across the warp)
      const float w = exp2f(ms - M[g]);
      L[g] = fmaf(w, __ldcg(a.part_ml + (it * G + g) * 2 + 1), L[g]);
      const float *po = a.part_o + (it * G + g) * D + lane * VPL;
#pragma unroll
      for (int e = 0; e < VPL; ++e) O[g][e] = fmaf(w, __ldcg(po + e), O[g][e]);
    }
  }
  T *out = reinterpret_cast<T *>(a.out) + ((size_t)i * a.H_q + (size_t)h * G) * D + lane * VPL;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float inv = L[g] > 0.f ? 1.f / L[g] : 0.f;
#pragma unroll
    for (int e = 0; e < VPL; ++e) Elem<T>::store(out + (size_t)g * D + e, O[g][e] * inv);
  }
}

// Take the unit's ticket after this warp's partial for one of its items is in memory; the
// holder of the last ticket merges.
template <typename T, int D, int G>
__device__ __forceinline__ void arrive(const DecodeArgs &a, int unit, int lane) {
  __threadfence();
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(a.tickets + unit, 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev == (unsigned)(a.n_items_max - 1)) {
    __threadfence();
    if (lane == 0) a.tickets[unit] = 0u;
    merge_unit<T, D, G>(a, unit, lane);
  }
}

template <int G>
__device__ __forceinline__ void write_empty_partial(const DecodeArgs &a, int item, int lane) {
  if (lane < G) {
    a.part_ml[((size_t)item * G + lane) * 2] = -INFINITY;
    a.part_ml[((size_t)item * G + lane) * 2 + 1] = 0.f;
  }
}

template <typename T, int D, int G, int NST>
__global__ void __launch_bounds__(32) decode_kernel(DecodeArgs a) {
  using TR = DT<T, D, G, NST>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stg = smem;
  float2 *pp = reinterpret_cast<float2 *>(smem + (size_t)NST * TR::STAGE);  // [16][G] (p, p)
  int4 *meta = reinterpret_cast<int4 *>(pp + 16 * G);                         // [NST]
  int *e_page = reinterpret_cast<int *>(meta + NST);                          // [kSwMax]
  int *e_blk = e_page + kSwMax;
  int *e_valid = e_blk + kSwMax;  // valid tokens of the entry's page, 0 = skip

  const int lane = threadIdx.x;
  const int tq = lane >> 3, dg = lane & 7;
  const int TW = gridDim.x;
  const int units = a.B * a.H_kv;
  const int total = units * a.n_items_max;
  const bool sparse = a.selected != nullptr;
  const T *kc = reinterpret_cast<const T *>(a.k_cache);
  const T *vc = reinterpret_cast<const T *>(a.v_cache);
  const T *qg = reinterpret_cast<const T *>(a.q);
  const size_t tok_stride = (size_t)a.H_kv * D;

  // ---- producer state -------------------------------------------------------------------
  int p_item = (int)blockIdx.x - TW;
  int p_unit = 0, p_e = 0, p_sub = 0, p_last = -1;
  bool p_has = false, p_first = false;

  // Advance the producer to its next item that has tiles; items without tiles are settled here.
  auto next_item = [&]() {
    p_has = false;
    for (;;) {
      p_item += TW;
      if (p_item >= total) return;
      const int unit = p_item / a.n_items_max;
      const int s = p_item - unit * a.n_items_max;
      const int i = unit / a.H_kv;
      const int L = a.seq_lens[i];
      const int P = (L + a.ps - 1) / a.ps;
      int nwin = 0;
      const int e0 = s * a.sw;
      if (L < 1 || P > a.max_pages) {
        if (s == 0 && lane == 0) set_status(a.ws, PSK_DEV_BAD_SEQLEN);
      } else {
        nwin = sparse ? min(a.sw, a.b_max - e0) : min(a.sw, P - e0);
      }
      int last_local = -1, first_local = kSwMax;
      const int32_t *row = sparse ? a.selected + (size_t)unit * a.b_max : nullptr;
      for (int e = lane; e < nwin; e += 32) {
        int page = e0 + e, blk = -1, valid = 0;
        bool ok = true;
        if (sparse) {
          page = row[e0 + e];
          const int prev = (e0 + e > 0) ? row[e0 + e - 1] : -1;
          if (page >= 0 && (page >= P || page <= prev || (e0 + e > 0 && prev < 0))) {
            set_status(a.ws, PSK_DEV_BAD_SELECTED);
            ok = false;
          }
          if (page < 0) ok = false;
        }
        if (ok) {
          blk = a.block_table[(size_t)i * a.max_pages + page];
          if (blk < 0 || blk >= a.nb) {
            set_status(a.ws, PSK_DEV_BAD_BLOCK);
            ok = false;
          }
        }
        if (ok) valid = min(a.ps, L - page * a.ps);
        e_page[e] = page;
        e_blk[e] = blk;
        e_valid[e] = valid;
        if (valid > 0) {
          last_local = max(last_local, e);
          first_local = min(first_local, e);
        }
      }
      const int last = warp_max_i(last_local);
      const int first = warp_min_i(first_local);
      __syncwarp();
      if (last < 0) {  // nothing to read in this item
        write_empty_partial<G>(a, p_item, lane);
        arrive<T, D, G>(a, unit, lane);
        continue;
      }
      p_unit = unit;
      p_e = first;
      p_sub = 0;
      p_last = last;
      p_first = true;
      p_has = true;
      return;
    }
  };

  // Issue the copies of the producer's next tile into `stage` (or an empty group).
  auto issue = [&](int stage) {
    int4 md = make_int4(-1, 0, 0, 0);
    if (p_has) {
      const int valid = e_valid[p_e];
      const int nv = min(16, valid - p_sub * 16);
      const size_t tok0 = (size_t)e_blk[p_e] * a.ps + p_sub * 16;
      const int h = p_unit % a.H_kv;
      const uint32_t sK = smem_u32(stg + (size_t)stage * TR::STAGE);
      const uint32_t sV = sK + TR::TILE;
#pragma unroll
      for (int u = 0; u < TR::LOADS; ++u) {
        const int q = lane + 32 * u;
        const int r = q / TR::NC, col = q - r * TR::NC;
        const bool ok = r < nv;
        const size_t goff = (tok0 + (ok ? r : 0)) * tok_stride + (size_t)h * D + (size_t)col * TR::EPC;
        cp_async16(sK + r * TR::ROW + col * 16, kc + goff, ok);
        cp_async16(sV + r * TR::ROW + col * 16, vc + goff, ok);
      }
      if (p_first) {
        const int i = p_unit / a.H_kv;
        const T *qrow = qg + ((size_t)i * a.H_q + (size_t)h * G) * D;
        const uint32_t sQ = sV + TR::TILE;
        for (int c = lane; c < TR::QCH; c += 32) cp_async16(sQ + c * 16, qrow + (size_t)c * TR::EPC, true);
      }
      // advance the cursor
      int flags = p_first ? 1 : 0;
      p_first = false;
      ++p_sub;
      if (p_sub * 16 >= valid) {
        p_sub = 0;
        do {
          ++p_e;
        } while (p_e <= p_last && e_valid[p_e] == 0);
      }
      const bool last = p_e > p_last;
      if (last) flags |= 2;
      md = make_int4(p_item, nv, flags, p_unit);
      if (last) next_item();
    }
    if (lane == 0) meta[stage] = md;
    cp_async_commit();
  };

  // ---- consumer state ---------------------------------------------------------------------
  float2 q2[G][TR::CPL * TR::EPC / 2];
  float m[G], l[G];
  float2 O[G][TR::VPL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < TR::VPL / 2; ++e) O[g][e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < TR::CPL * TR::EPC / 2; ++e) q2[g][e] = make_float2(0.f, 0.f);
  }

  next_item();
#pragma unroll
  for (int st = 0; st < NST - 1; ++st) issue(st);
  int stage = 0;
  for (;;) {
    issue((stage + NST - 1) % NST);
    cp_async_wait<NST - 1>();
    __syncwarp();
    const int4 md = meta[stage];
    if (md.x < 0) break;  // the producer ran out: every later stage is empty too
    const int nv = md.y;
    const unsigned char *sK = stg + (size_t)stage * TR::STAGE;
    const unsigned char *sV = sK + TR::TILE;
    if (md.z & 1) {  // first tile of an item: its q rows came with it
      const unsigned char *sQ = sV + TR::TILE;
      const float qs = a.scale * kLog2e;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < TR::CPL; ++c) {
          float2 f[TR::EPC / 2];
          Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(sQ + g * TR::ROW + (dg + 8 * c) * 16), f);
#pragma unroll
          for (int e = 0; e < TR::EPC / 2; ++e) q2[g][c * TR::EPC / 2 + e] = make_float2(f[e].x * qs, f[e].y * qs);
        }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < TR::VPL / 2; ++e) O[g][e] = make_float2(0.f, 0.f);
      }
    }
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
            for (int e = 0; e < TR::EPC / 2; ++e) acc[tt][g] = ffma2(q2[g][c * TR::EPC / 2 + e], kf[e], acc[tt][g]);
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
    for (int tk = 0; tk < nv; ++tk) {
      float2 vf[TR::VPL / 2];
      const unsigned char *vr = sV + tk * TR::ROW + lane * TR::VPL * TR::ES;
      if constexpr (TR::VPL * TR::ES == 16) {
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
    }
    if (md.z & 2) {  // the item's last tile: write its partial, take the unit's ticket
      const size_t item = (size_t)md.x;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float lg = warp_sum(l[g]);
        float2 *po = reinterpret_cast<float2 *>(a.part_o + (item * G + g) * D + lane * TR::VPL);
#pragma unroll
        for (int e = 0; e < TR::VPL / 2; ++e) po[e] = O[g][e];
        if (lane == 0) {
          a.part_ml[(item * G + g) * 2] = m[g];
          a.part_ml[(item * G + g) * 2 + 1] = lg;
        }
      }
      arrive<T, D, G>(a, md.w, lane);
    }
    __syncwarp();
    stage = (stage + 1) % NST;
  }
  cp_async_wait<0>();
}

template <typename T, int D, int G>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t s) {
  constexpr int NST = 3;
  using TR = DT<T, D, G, NST>;
  auto kfn = decode_kernel<T, D, G, NST>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TR::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, 32, TR::SMEM)) != cudaSuccess) return e;
  const long long items = (long long)a.B * a.H_kv * a.n_items_max;
  const int grid = (int)std::max(1LL, std::min<long long>((long long)sms * std::max(1, per_sm), items));
  kfn<<<grid, 32, TR::SMEM, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool plan_decode(const psk_layout &L, int entries, bool dense, DecodePlan *plan) {
  const long long units = (long long)L.batch * L.num_kv_heads;
  // aim at ~8 items per warp of a full persistent grid (152 SMs x ~7 warps)
  const long long target_items = 8LL * 152 * 7;
  const long long sw = (units * entries) / target_items;
  int p2 = 1;
  while (p2 * 2 <= sw && p2 < kSwMax) p2 *= 2;
  plan->sw = std::max(dense ? 4 : 2, p2);
  plan->n_items_max = (entries + plan->sw - 1) / plan->sw;
  const int G = L.num_q_heads / L.num_kv_heads;
  size_t off = ws_scratch_offset((size_t)units);
  plan->off_o = off;
  off = align_up(off + (size_t)units * plan->n_items_max * G * L.v_head_dim * 4, 256);
  plan->off_ml = off;
  off = align_up(off + (size_t)units * plan->n_items_max * G * 2 * 4, 256);
  plan->ws_bytes = off;
  plan->off_tickets = ws_decode_tickets_offset((size_t)units);
  return (long long)units * plan->n_items_max < (1LL << 31);
}

#define PSK_DECODE_CASES(X)   \
  X(bf16_t, PSK_BF16, 128, 4) \
  X(bf16_t, PSK_BF16, 64, 4)  \
  X(float, PSK_F32, 64, 4)    \
  X(float, PSK_F32, 128, 4)

bool decode_supported(int dtype, int D, int D_v, int G, int ps) {
  if (D_v != D || ps % 16 != 0 || ps > 16 * kSwMax) return false;
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
