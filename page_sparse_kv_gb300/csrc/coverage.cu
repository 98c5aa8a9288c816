// Adaptive per-head coverage over exact page masses (LOCKS PKG-INFO, "Configuration
// (LocksConfig)", `coverage`: adaptive per-head nucleus coverage over exact page masses, GQA;
// AMASS PyPI page, "Key AmassConfig fields", the same option, default 0.95).
//
// A page's mass for query head g is the softmax weight of its tokens among all the sequence's
// tokens; a KV head's page mass is the max over its group (the group combine `max`). The unit's
// selection is its always-kept pages plus the fewest other pages, highest mass first (ties to
// the lower page), whose mass with the always-kept pages' reaches `coverage` times the unit's
// total mass, capped at b_max pages. Three launches:
//
//   page_mass_kernel      a K-only pass over every page: per (unit, page, query head) the max
//                         m and the sum s = sum_t 2^(x_t - m) of the page's logits x_t =
//                         scale * log2(e) * q . k_t (fp32).
//   coverage_keys_kernel  one CTA per unit: the group's normalisers M_g = max_p m, Z_g =
//                         sum_p s 2^(m - M_g); each page's mass max_g s 2^(m - M_g) / Z_g;
//                         the selection key of that mass (0 for an always-kept page); and the
//                         nucleus size k. The masses are summed as 40-bit fixed-point integers
//                         (order-independent); an MSB-first radix pass over the keys with a
//                         count and a mass histogram per 8-bit digit finds the key T where the
//                         running mass of the keys above it crosses the target; every key equal
//                         to T carries the same mass, so the number of them needed follows.
//                         The unit's budget is |always kept| + min(k, b_max - |always kept|).
//   page_select_kernel    (select.cu) top-b by those keys with that per-unit budget.
#include <algorithm>

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMassThreads = 128;  // four warps, one page at a time each
constexpr int kMassPages = 32;     // pages per CTA of the mass pass
constexpr int kCovThreads = 256;
constexpr double kMassQuant = 1099511627776.0;  // 2^40: fixed-point unit of a page mass

// ---- K-only pass ----------------------------------------------------------------------------
// Grid (page chunk, unit). Lane layout for a row of D elements: LPR = D * ES / 16 lanes, one
// 16-byte chunk each; RPW = 32 / LPR rows per warp step.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kMassThreads) page_mass_kernel(CoverageArgs a) {
  pdl_begin();
  constexpr int EPC = Elem<T>::kPerChunk;
  constexpr int LPR = D / EPC;
  constexpr int RPW = 32 / LPR;
  static_assert(LPR >= 1 && LPR <= 32 && (LPR & (LPR - 1)) == 0, "row of 16..512 bytes, power of 2");
  const int unit = blockIdx.y;
  const int i = unit / a.H_kv, h = unit - i * a.H_kv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by coverage_keys_kernel
  const int sub = lane % LPR, rg = lane / LPR;
  // q slices of this lane for the G heads of the group, scaled into the log2 domain
  float2 q2[G][EPC / 2];
  {
    const T *qb = reinterpret_cast<const T *>(a.q) + ((size_t)i * a.H_q + (size_t)h * G) * D + sub * EPC;
    const float qs = a.scale * kLog2e;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float2 f[EPC / 2];
      Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(qb + (size_t)g * D), f);
#pragma unroll
      for (int e = 0; e < EPC / 2; ++e) q2[g][e] = make_float2(f[e].x * qs, f[e].y * qs);
    }
  }
  const T *kc = reinterpret_cast<const T *>(a.k_cache);
  const size_t row_stride = (size_t)a.H_kv * D;
  for (int p = blockIdx.x * kMassPages + warp; p < min(P, (blockIdx.x + 1) * kMassPages); p += kMassThreads / 32) {
    const int blk = a.block_table[(size_t)i * a.max_pages + p];
    float m[G], s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      s[g] = 0.f;
    }
    if (blk < 0 || blk >= a.nb) {
      if (lane == 0) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    } else {
      const int nv = min(a.ps, seq_len - p * a.ps);
      const T *base = kc + ((size_t)blk * a.ps) * row_stride + (size_t)h * D + sub * EPC;
      for (int r0 = 0; r0 < nv; r0 += RPW) {
        const int r = r0 + rg;
        float x[G];
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r < nv) w = __ldcs(reinterpret_cast<const uint4 *>(base + (size_t)r * row_stride));
        float2 kf[EPC / 2];
        Elem<T>::to_f2(w, kf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < EPC / 2; ++e) acc = ffma2(q2[g][e], kf[e], acc);
          x[g] = acc.x + acc.y;
        }
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) x[g] += __shfl_xor_sync(0xffffffffu, x[g], o);
        if (r < nv) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float mn = fmaxf(m[g], x[g]);
            s[g] = s[g] * exp2f(m[g] - mn) + exp2f(x[g] - mn);
            m[g] = mn;
          }
        }
      }
      // combine the RPW row groups (lanes that differ in the row-group bits)
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mo = __shfl_xor_sync(0xffffffffu, m[g], o);
          const float so = __shfl_xor_sync(0xffffffffu, s[g], o);
          const float mn = fmaxf(m[g], mo);
          s[g] = (m[g] == -INFINITY ? 0.f : s[g] * exp2f(m[g] - mn)) + (mo == -INFINITY ? 0.f : so * exp2f(mo - mn));
          m[g] = mn;
        }
    }
    if (lane < G) {
      float mg = m[0], sg = s[0];
#pragma unroll
      for (int g = 1; g < G; ++g)
        if (g == lane) {
          mg = m[g];
          sg = s[g];
        }
      float *dst = a.pm + (((size_t)unit * a.max_pages + p) * G + lane) * 2;
      dst[0] = mg;
      dst[1] = sg;
    }
  }
}

// ---- per-unit normalisation, keys and nucleus size -----------------------------------------
__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kCovThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < kCovThreads / 32; ++w) r += red[w];
  return r;
}
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned long long r = 0;
#pragma unroll
  for (int w = 0; w < kCovThreads / 32; ++w) r += red[w];
  return r;
}

template <int G>
__global__ void __launch_bounds__(kCovThreads) coverage_keys_kernel(CoverageArgs a) {
  pdl_wait();  // dependents are released when this grid completes
  __shared__ float redf[kCovThreads / 32];
  __shared__ unsigned long long redu[kCovThreads / 32];
  __shared__ unsigned long long hmass[256];
  __shared__ int hcount[256];
  __shared__ int pick[3];
  __shared__ unsigned long long pick_mass[2];
  const int unit = blockIdx.x;
  const int i = unit / a.H_kv;
  const int tid = threadIdx.x;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) {
    if (tid == 0) {
      set_status(a.ws, PSK_DEV_BAD_SEQLEN);
      a.unit_budgets[unit] = 0;  // the selection writes the row as -1
    }
    return;
  }
  const float *pm = a.pm + (size_t)unit * a.max_pages * G * 2;
  float M[G], Zinv[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mx = -INFINITY;
    for (int p = tid; p < P; p += kCovThreads) mx = fmaxf(mx, pm[(p * G + g) * 2]);
    M[g] = block_max(mx, redf);
    float z = 0.f;
    for (int p = tid; p < P; p += kCovThreads) {
      const float m = pm[(p * G + g) * 2];
      if (m != -INFINITY) z += pm[(p * G + g) * 2 + 1] * exp2f(m - M[g]);
    }
    const float Z = block_sum(z, redf);
    Zinv[g] = Z > 0.f ? 1.f / Z : 0.f;
  }
  // page masses, keys, fixed-point masses
  uint32_t *krow = a.keys + (size_t)unit * a.key_stride;
  unsigned long long *qrow = a.qmass + (size_t)unit * a.max_pages;
  unsigned long long forced_q = 0, total_q = 0;
  int n_cand = 0;
  for (int p = tid; p < P; p += kCovThreads) {
    float mass = 0.f;
    bool read = false;  // false only for a page whose block id was out of range (flagged)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m = pm[(p * G + g) * 2];
      if (m != -INFINITY) {
        read = true;
        mass = fmaxf(mass, pm[(p * G + g) * 2 + 1] * exp2f(m - M[g]) * Zinv[g]);
      }
    }
    const unsigned long long qm = (unsigned long long)((double)mass * kMassQuant + 0.5);
    if (a.masses_out) a.masses_out[(size_t)unit * a.max_pages + p] = mass;
    const bool forced = always_kept(p, P, a.sink, a.window);
    krow[p] = (forced || !read) ? 0u : score_key(mass);
    qrow[p] = qm;
    total_q += qm;
    if (forced) forced_q += qm;
    else if (read) ++n_cand;
  }
  total_q = block_sum_u64(total_q, redu);
  forced_q = block_sum_u64(forced_q, redu);
  n_cand = (int)block_sum_u64((unsigned long long)n_cand, redu);
  __syncthreads();  // keys and masses of the row are written (each thread reads back any of them)
  const unsigned long long target = (unsigned long long)ceil((double)total_q * a.coverage);
  int k = 0;
  if (forced_q < target && n_cand > 0) {
    unsigned long long need = target - forced_q;  // mass still to cover
    int taken = 0;                                // keys above the running prefix
    uint32_t prefix = 0u, mask = 0u;
    bool all = false;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int x = tid; x < 256; x += kCovThreads) {
        hmass[x] = 0ull;
        hcount[x] = 0;
      }
      __syncthreads();
      for (int p = tid; p < P; p += kCovThreads) {
        const uint32_t key = krow[p];
        if (key != 0u && (key & mask) == prefix) {
          atomicAdd(&hmass[(key >> shift) & 255u], qrow[p]);
          atomicAdd(&hcount[(key >> shift) & 255u], 1);
        }
      }
      __syncthreads();
      if (tid == 0) {
        // descending digits: the first whose running mass reaches what is still needed
        unsigned long long run = 0;
        int cnt = 0, d = -1;
        for (int b = 255; b >= 0; --b) {
          if (run + hmass[b] >= need && hcount[b] > 0) {
            d = b;
            break;
          }
          run += hmass[b];
          cnt += hcount[b];
        }
        pick[0] = d;
        pick[1] = cnt;
        pick[2] = d >= 0 ? hcount[d] : 0;
        pick_mass[0] = run;
        pick_mass[1] = d >= 0 ? hmass[d] : 0ull;
      }
      __syncthreads();
      const int d = pick[0];
      if (d < 0) {  // the candidates' mass falls short of the target (rounding): take them all
        all = true;
        break;
      }
      need -= pick_mass[0];
      taken += pick[1];
      prefix |= (uint32_t)d << shift;
      mask |= 255u << shift;
      if (shift == 0) {
        // every key equal to prefix has the same mass: how many of them make up `need`
        const unsigned long long each = pick_mass[1] / (unsigned long long)pick[2];
        const unsigned long long n_eq = each > 0 ? (need + each - 1) / each : (unsigned long long)pick[2];
        taken += (int)min((unsigned long long)pick[2], max(1ull, n_eq));
      }
      __syncthreads();  // pick is rewritten by the next pass
    }
    k = all ? n_cand : taken;
  }
  if (tid == 0) {
    const int n_forced = min(P, a.sink + a.window);
    a.unit_budgets[unit] = n_forced + min(k, max(0, a.b_max - n_forced));
  }
}

template <typename T, int D, int G>
cudaError_t launch_t(const CoverageArgs &c, const ScoreArgs &sel, cudaStream_t s) {
  dim3 g1((c.max_pages + kMassPages - 1) / kMassPages, c.B * c.H_kv);
  cudaError_t e = launch_kernel(true, page_mass_kernel<T, D, G>, g1, kMassThreads, 0, s, c);
  if (e != cudaSuccess) return e;
  e = launch_kernel(false, coverage_keys_kernel<G>, c.B * c.H_kv, kCovThreads, 0, s, c);
  if (e != cudaSuccess) return e;
  return launch_page_select(sel, s);
}

}  // namespace

#define PSK_COVERAGE_CASES(X) \
  X(bf16_t, PSK_BF16, 128, 4) \
  X(bf16_t, PSK_BF16, 64, 4)  \
  X(float, PSK_F32, 64, 4)    \
  X(float, PSK_F32, 128, 4)   \
  X(bf16_t, PSK_BF16, 128, 1) \
  X(bf16_t, PSK_BF16, 128, 2) \
  X(bf16_t, PSK_BF16, 64, 1)  \
  X(bf16_t, PSK_BF16, 64, 2)  \
  X(float, PSK_F32, 64, 1)    \
  X(float, PSK_F32, 128, 1)

bool coverage_supported(int dtype, int D, int G) {
#define X(TT, DT, DD, GG) \
  if (dtype == DT && D == DD && G == GG) return true;
  PSK_COVERAGE_CASES(X)
#undef X
  return false;
}

cudaError_t launch_coverage_select(const CoverageArgs &c, const ScoreArgs &sel, int dtype, cudaStream_t s) {
  const int G = c.H_q / c.H_kv;
#define X(TT, DT, DD, GG) \
  if (dtype == DT && c.D == DD && G == GG) return launch_t<TT, DD, GG>(c, sel, s);
  PSK_COVERAGE_CASES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace psk
