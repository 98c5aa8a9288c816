// Stage 4: exact softmax attention over the selected pages of a GQA paged cache, split-K
// over pages with an fp32 online-softmax (m, l, O) state and a log-sum-exp combine
// (EntmaxKV README, introduction: "the attention is exact over that selection"; LOCKS
// PKG-INFO, "How it works", Sparse decode: a paged kernel that reads only the selected
// pages). The dense decode is the same kernel with the implicit list 0 .. P-1.
//
// Work decomposition: one CTA of NW warps per (split of `split` list entries, KV head,
// sequence). The group's G query heads share every K/V element loaded, so each element is
// converted once and used G times. A page is cut into 16-token tiles; warp w takes tiles
// w, w + NW, ... of the split and keeps its own (m, l, O) state. Tiles are staged into a
// per-warp ring of NST shared-memory stages with 16-byte cp.async (zero fill for rows past
// seq_len, so masked rows never carry stale data into P.V), NST - 1 tiles in flight.
//
// Per tile and warp: lane = (tq = lane / 8, dg = lane % 8). QK: the lane owns the 16-byte
// chunks dg, dg + 8, ... of each K row and the matching q slices (pre-scaled by
// scale * log2(e) so exp2 gives the softmax weights), and computes partial dot products
// for tokens tq, tq + 4, tq + 8, tq + 12 and all G heads with packed fp32x2 FMAs; a
// transposing butterfly over the 8 dg lanes leaves each lane with full logits of one token
// for G/2 heads. Softmax: tile max per head by 4 shuffles, online rescale, p to a per-warp
// shared array. PV: lane owns D/32 output dims for all G heads and reads one V row chunk
// per token (conflict-free 8-byte loads) plus the G broadcast p values.
//
// At the end the NW warp states are merged through shared memory into one partial per
// CTA (m, l and the unnormalised O relative to m); the combine kernel merges the splits
// of each (sequence, KV head) by log-sum-exp and writes out in the storage dtype.
#include <algorithm>

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplit = 64;

template <typename T, int D, int G, int NW, int NST>
struct DecodeTraits {
  static constexpr int ES = Elem<T>::kBytes;
  static constexpr int EPC = Elem<T>::kPerChunk;  // elements per 16-byte chunk
  static constexpr int NC = D / EPC;               // chunks per row
  static constexpr int CPL = NC / 8;               // QK chunks per lane
  static constexpr int VPL = D / 32;               // PV dims per lane
  static constexpr int ROW = D * ES;               // bytes per row
  static constexpr int TILE_BYTES = 16 * ROW;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile + V tile
  static constexpr int LOADS = 16 * NC / 32;          // 16-byte chunks per lane per tile (K)
  static constexpr int NV = 4 * G;                    // partial logits per lane before reduce
  static constexpr int KEEP = NV >= 8 ? NV / 8 : 1;   // logits per lane after reduce
  static constexpr size_t SMEM = (size_t)NW * NST * STAGE_BYTES  // stages
                                 + (size_t)NW * 16 * G * 4       // p values
                                 + (size_t)NW * G * D * 4        // warp O for the merge
                                 + (size_t)NW * G * 2 * 4        // warp m, l
                                 + (size_t)kMaxSplit * 3 * 4;    // entry table
  static_assert(NC % 8 == 0, "a row must be a multiple of 128 bytes");
  static_assert(D % 32 == 0, "head_dim must be a multiple of 32");
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

template <typename T, int D, int G, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) decode_split_kernel(DecodeArgs a) {
  using TR = DecodeTraits<T, D, G, NW, NST>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stages = smem;
  float *p_sh = reinterpret_cast<float *>(smem + (size_t)NW * NST * TR::STAGE_BYTES);
  float *wO = p_sh + NW * 16 * G;
  float *wML = wO + NW * G * D;
  int *ent_page = reinterpret_cast<int *>(wML + NW * G * 2);
  int *ent_blk = ent_page + kMaxSplit;
  int *ent_valid = ent_blk + kMaxSplit;

  const int s = blockIdx.x, h = blockIdx.y, i = blockIdx.z;
  const int unit = i * a.H_kv + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tq = lane >> 3, dg = lane & 7;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  const int e0 = s * a.split;

  // ---- entries of this split -------------------------------------------------------------
  int n_ent;
  if (seq_len < 1 || P > a.max_pages) {
    if (s == 0 && tid == 0) set_status(a.ws, PSK_DEV_BAD_SEQLEN);
    n_ent = 0;
  } else if (a.selected) {
    const int32_t *row = a.selected + (size_t)unit * a.b_max;
    if (e0 >= a.b_max || row[e0] < 0) return;  // the combine skips this split too
    n_ent = min(a.split, a.b_max - e0);
  } else {
    if (e0 >= P) return;
    n_ent = min(a.split, P - e0);
  }
  if (tid < n_ent) {
    int p = e0 + tid, blk = -1, valid = 0;
    bool ok = true;
    if (a.selected) {
      const int32_t *row = a.selected + (size_t)unit * a.b_max;
      p = row[e0 + tid];
      const int prev = (e0 + tid > 0) ? row[e0 + tid - 1] : -1;
      if (p >= 0 && (p >= P || p <= prev || (e0 + tid > 0 && prev < 0))) {
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
    valid = ok ? min(a.ps, seq_len - p * a.ps) : 0;
    ent_page[tid] = p;
    ent_blk[tid] = blk;
    ent_valid[tid] = valid;
  }
  __syncthreads();

  // ---- per-lane query slices (scaled into the log2 domain) --------------------------------
  float2 q2[G][TR::CPL * TR::EPC / 2];
  {
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

  float m[G], l[G], O[G][TR::VPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < TR::VPL; ++e) O[g][e] = 0.f;
  }

  const int stp = a.ps / 16;  // tiles per page
  const int ntiles = n_ent * stp;
  unsigned char *my_stages = stages + (size_t)warp * NST * TR::STAGE_BYTES;
  float *my_p = p_sh + warp * 16 * G;
  const T *kc = reinterpret_cast<const T *>(a.k_cache);
  const T *vc = reinterpret_cast<const T *>(a.v_cache);
  const size_t head_off = (size_t)h * D;
  const size_t tok_stride = (size_t)a.H_kv * D;

  auto tile_rows = [&](int it) -> int {
    const int e = it / stp, sub = it - e * stp;
    return min(16, ent_valid[e] - sub * 16);
  };
  auto load_tile = [&](int it, int stage) {
    if (it < ntiles) {
      const int e = it / stp, sub = it - e * stp;
      const int nv = min(16, ent_valid[e] - sub * 16);
      if (nv > 0) {
        const size_t tok0 = (size_t)ent_blk[e] * a.ps + sub * 16;
        const uint32_t sK = smem_u32(my_stages + (size_t)stage * TR::STAGE_BYTES);
        const uint32_t sV = sK + TR::TILE_BYTES;
#pragma unroll
        for (int u = 0; u < TR::LOADS; ++u) {
          const int q = lane + 32 * u;
          const int r = q / TR::NC, col = q - r * TR::NC;
          const bool ok = r < nv;
          const size_t goff = (tok0 + (ok ? r : 0)) * tok_stride + head_off + (size_t)col * TR::EPC;
          cp_async16(sK + r * TR::ROW + col * 16, kc + goff, ok);
          cp_async16(sV + r * TR::ROW + col * 16, vc + goff, ok);
        }
      }
    }
    cp_async_commit();
  };

  int next = warp;
#pragma unroll
  for (int st = 0; st < NST - 1; ++st) {
    load_tile(next, st);
    next += NW;
  }
  int stage = 0;
  for (int cur = warp; cur < ntiles; cur += NW) {
    load_tile(next, (stage + NST - 1) % NST);
    next += NW;
    cp_async_wait<NST - 1>();
    __syncwarp();
    const int nv = tile_rows(cur);
    if (nv > 0) {
      const unsigned char *sK = my_stages + (size_t)stage * TR::STAGE_BYTES;
      const unsigned char *sV = sK + TR::TILE_BYTES;
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
      // lane now holds token t for heads hb*KEEP + j  (G >= 2), or head 0 (G == 1)
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
      float alpha[G], mnew[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int j = g % TR::KEEP, half = g / TR::KEEP;
        const float tmax = (G == 1 || half == hb) ? mx[j] : oth[j];
        mnew[g] = fmaxf(m[g], tmax);
        alpha[g] = exp2f(m[g] - mnew[g]);
        m[g] = mnew[g];
        l[g] *= alpha[g];
#pragma unroll
        for (int e = 0; e < TR::VPL; ++e) O[g][e] *= alpha[g];
      }
      const bool writer = (G >= 2) || ((dg & 1) == 0);
#pragma unroll
      for (int j = 0; j < TR::KEEP; ++j) {
        const int gj = hb * TR::KEEP + j;
        float mg = mnew[0];
#pragma unroll
        for (int g = 1; g < G; ++g)
          if (g == gj) mg = mnew[g];
        const float p = exp2f(v[j] - mg);
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g == gj && writer) l[g] += p;
        if (writer) my_p[t * G + gj] = p;
      }
      __syncwarp();
      // ---- PV ----
      for (int tk = 0; tk < nv; ++tk) {
        float vf[TR::VPL];
        const unsigned char *vr = sV + tk * TR::ROW + lane * TR::VPL * TR::ES;
        if constexpr (TR::VPL * TR::ES == 16) {
          float2 f[TR::VPL / 2];
          Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(vr), f);
#pragma unroll
          for (int e = 0; e < TR::VPL / 2; ++e) {
            vf[2 * e] = f[e].x;
            vf[2 * e + 1] = f[e].y;
          }
        } else if constexpr (TR::VPL * TR::ES == 8) {
          float2 f[TR::VPL / 2];
          Elem<T>::to_f2_8(*reinterpret_cast<const uint2 *>(vr), f);
#pragma unroll
          for (int e = 0; e < TR::VPL / 2; ++e) {
            vf[2 * e] = f[e].x;
            vf[2 * e + 1] = f[e].y;
          }
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t *>(vr);
          vf[0] = bf16_lo(w);
          vf[1] = bf16_hi(w);
        }
        const float *pr = my_p + tk * G;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = pr[g];
#pragma unroll
          for (int e = 0; e < TR::VPL; ++e) O[g][e] = fmaf(pg, vf[e], O[g][e]);
        }
      }
    }
    __syncwarp();
    stage = (stage + 1) % NST;
  }
  cp_async_wait<0>();

  // ---- merge the warps of the CTA --------------------------------------------------------
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float x = l[g];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    l[g] = x;
#pragma unroll
    for (int e = 0; e < TR::VPL; ++e) wO[(warp * G + g) * D + lane * TR::VPL + e] = O[g][e];
    if (lane == 0) {
      wML[(warp * G + g) * 2] = m[g];
      wML[(warp * G + g) * 2 + 1] = l[g];
    }
  }
  __syncthreads();
  const size_t pbase = (size_t)unit * a.n_splits_max + s;
  for (int idx = tid; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
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
    a.part_o[(pbase * G + g) * D + d] = acc;
    if (d == 0) {
      a.part_ml[(pbase * G + g) * 2] = M;
      a.part_ml[(pbase * G + g) * 2 + 1] = L;
    }
  }
}

// One CTA per (sequence, KV head): merge its splits and write G output rows.
template <typename T, int G>
__global__ void combine_kernel(DecodeArgs a) {
  const int unit = blockIdx.x;
  const int i = unit / a.H_kv, h = unit - i * a.H_kv;
  const int D = a.D_v;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  const bool bad = seq_len < 1 || P > a.max_pages;
  const int32_t *row = a.selected ? a.selected + (size_t)unit * a.b_max : nullptr;
  T *out = reinterpret_cast<T *>(a.out) + ((size_t)i * a.H_q + (size_t)h * G) * D;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, d = idx - g * D;
    float M = -INFINITY;
    for (int s = 0; s < a.n_splits_max; ++s) {
      const int e0 = s * a.split;
      const bool live = !bad && (row ? (e0 < a.b_max && row[e0] >= 0) : e0 < P);
      if (!live) break;
      M = fmaxf(M, a.part_ml[(((size_t)unit * a.n_splits_max + s) * G + g) * 2]);
    }
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < a.n_splits_max; ++s) {
        const int e0 = s * a.split;
        const bool live = row ? (e0 < a.b_max && row[e0] >= 0) : e0 < P;
        if (!live) break;
        const size_t b = ((size_t)unit * a.n_splits_max + s) * G + g;
        const float sc = exp2f(a.part_ml[b * 2] - M);
        acc = fmaf(sc, a.part_o[b * D + d], acc);
        L = fmaf(sc, a.part_ml[b * 2 + 1], L);
      }
    }
    Elem<T>::store(out + (size_t)g * D + d, L > 0.f ? acc / L : 0.f);
  }
}

template <typename T, int D, int G>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t s) {
  constexpr int NW = 4, NST = 3;
  using TR = DecodeTraits<T, D, G, NW, NST>;
  auto kfn = decode_split_kernel<T, D, G, NW, NST>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TR::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_splits_max, a.H_kv, a.B);
  kfn<<<grid, NW * 32, TR::SMEM, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  combine_kernel<T, G><<<a.B * a.H_kv, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool plan_decode(const psk_layout &L, int entries, bool dense, DecodePlan *plan) {
  const long long units = (long long)L.batch * L.num_kv_heads;
  int split = dense ? 32 : 16;
  // shrink the split while the grid would not fill the GPU twice over (152 SMs x 2 CTAs)
  while (split > 4 && units * ((entries + split - 1) / split) < 2 * 152 * 2) split /= 2;
  // a page of page_size tokens is page_size / 16 tiles; keep tiles per CTA bounded
  plan->split = std::min(split, kMaxSplit);
  plan->n_splits_max = (entries + plan->split - 1) / plan->split;
  const int G = L.num_q_heads / L.num_kv_heads;
  size_t off = ws_scratch_offset((size_t)units);
  plan->off_o = off;
  off = align_up(off + (size_t)units * plan->n_splits_max * G * L.v_head_dim * 4, 256);
  plan->off_ml = off;
  off = align_up(off + (size_t)units * plan->n_splits_max * G * 2 * 4, 256);
  plan->ws_bytes = off;
  return plan->n_splits_max <= 65535;
}

#define PSK_DECODE_CASES(X)   \
  X(bf16_t, PSK_BF16, 128, 4) \
  X(bf16_t, PSK_BF16, 64, 4)  \
  X(float, PSK_F32, 64, 4)    \
  X(float, PSK_F32, 128, 4)

bool decode_supported(int dtype, int D, int D_v, int G, int ps) {
  if (D_v != D || ps % 16 != 0 || ps > 64) return false;
#define X(TT, DT, DD, GG) \
  if (dtype == DT && D == DD && G == GG) return true;
  PSK_DECODE_CASES(X)
#undef X
  return false;
}

cudaError_t launch_decode(const DecodeArgs &a, int dtype, cudaStream_t s) {
  const int D = a.D, G = a.H_q / a.H_kv;
#define X(TT, DT, DD, GG) \
  if (dtype == DT && D == DD && G == GG) return launch_t<TT, DD, GG>(a, s);
  PSK_DECODE_CASES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace psk
