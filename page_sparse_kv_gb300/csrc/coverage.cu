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
//                         scale * log2(e) * q . k_t (fp32). bf16 caches take
//                         page_mass_mma_kernel instead: the same sums with q . k on the tensor
//                         cores, K staged by TMA (unless PSK_DECODE_MMA=0).
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
constexpr int kCovHist = 8;        // histogram copies of the nucleus search
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

// ---- K-only pass on the tensor cores (bf16) -------------------------------------------------
// Grid (page chunk, unit), four warps; warp w takes pages w, w + 4, ... of the chunk. Each page's
// 16-token K tiles stream through the warp's two-stage TMA ring as 128-byte boxes stored with
// the 128-byte swizzle (the decode's tile layout), and S = q K^T is D/16 k-steps of one
// ldmatrix and two mma.sync m16n8k16 with the G query heads as the M rows. Lane (g = lane / 4,
// t4 = lane % 4) holds the logits of tokens 2 t4, 2 t4 + 1, 8 + 2 t4, 9 + 2 t4 for head g; the
// page's (m, s) per head is an online max / sum over its tiles, reduced over the row's 4 lanes
// when the page ends. Rows past seq_len may hold anything: their logits are set to -inf.
constexpr int kMassMmaWarps = 4;
constexpr int kMassStages = 2;

template <int D>
constexpr size_t mass_mma_smem() {
  return 1024 + (size_t)kMassMmaWarps * kMassStages * 16 * D * 2;
}

template <int D, int G>
__global__ void __launch_bounds__(kMassMmaWarps * 32) page_mass_mma_kernel(CoverageArgs a,
                                                                           const __grid_constant__ CUtensorMap tmK) {
  pdl_begin();
  static_assert(G >= 1 && G <= 8, "query heads are the MMA rows 0..7");
  constexpr int KS = D / 16;          // k-steps of q K^T
  constexpr int TILE = 16 * D * 2;    // one K tile: 16 rows
  constexpr int BOX = 16 * 128;       // one 128-byte box of 16 rows
  constexpr int NB = D * 2 / 128;     // boxes per row
  extern __shared__ unsigned char mass_dyn[];
  unsigned char *base =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(mass_dyn) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[kMassMmaWarps][kMassStages];
  const int unit = blockIdx.y;
  const int i = unit / a.H_kv, h = unit - i * a.H_kv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by coverage_keys_kernel
  const int pc0 = blockIdx.x * kMassPages, pc1 = min(P, pc0 + kMassPages);
  if (pc0 >= pc1) return;
  const int stp = a.ps / 16;  // tiles per page
  const int n_pages = pc1 - pc0 > warp ? (pc1 - pc0 - warp + kMassMmaWarps - 1) / kMassMmaWarps : 0;
  const int ntiles = n_pages * stp;
  unsigned char *my = base + (size_t)warp * kMassStages * TILE;
  if (lane == 0) {
    for (int k = 0; k < kMassStages; ++k) mbar_init(smem_u32(&bars[warp][k]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  // tile k of this warp: page pc0 + warp + (k / stp) * 4, 16-row slice k % stp
  auto tile_page = [&](int k) { return pc0 + warp + (k / stp) * kMassMmaWarps; };
  auto tile_rows = [&](int k) {
    const int p = tile_page(k), sub = k % stp;
    return min(16, seq_len - p * a.ps - sub * 16);
  };
  auto tile_blk = [&](int k) { return a.block_table[(size_t)i * a.max_pages + tile_page(k)]; };
  auto issue = [&](int k) {
    if (k >= ntiles || lane != 0) return;
    const int stg = k % kMassStages;
    const uint32_t bar = smem_u32(&bars[warp][stg]);
    const int blk = tile_blk(k), nv = tile_rows(k);
    if (nv > 0 && blk >= 0 && blk < a.nb) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, TILE);
      const uint32_t dst = smem_u32(my + (size_t)stg * TILE);
      const int row = blk * a.ps + (k % stp) * 16;
      const uint64_t pol = l2_evict_first_policy();  // read once
#pragma unroll
      for (int b = 0; b < NB; ++b) tma_load_3d_stream(dst + b * BOX, &tmK, b * 64, h, row, bar, pol);
    } else {
      mbar_arrive_expect_tx(bar, 0u);
    }
  };
  for (int k = 0; k < kMassStages - 1; ++k) issue(k);

  const int g = lane >> 2, t4 = lane & 3, r8 = lane & 7, mi = lane >> 3;
  uint32_t qa[KS][2];  // q as the A operand (rows 0..G-1; rows 8..15 zero)
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
  const float qs = a.scale * kLog2e;
  const int k_tok = (mi >> 1) * 8 + r8, k_ch = mi & 1;
  float m_run = -INFINITY, s_run = 0.f;  // row g's running (max, this lane's share of the sum)
  for (int k = 0; k < ntiles; ++k) {
    issue(k + kMassStages - 1);
    const int stg = k % kMassStages;
    mbar_wait(smem_u32(&bars[warp][stg]), (k / kMassStages) & 1, a.ws);
    const int blk = tile_blk(k), nv = tile_rows(k);
    const bool ok = blk >= 0 && blk < a.nb;
    if (!ok && lane == 0 && k % stp == 0) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    if (ok && nv > 0) {
      const uint32_t aK = smem_u32(my + (size_t)stg * TILE);
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int ch = 2 * s + k_ch;
        uint32_t kb[4];
        ldsm_x4(aK + (ch >> 3) * BOX + k_tok * 128 + (((ch & 7) ^ r8) << 4), kb);
        const uint32_t qa4[4] = {qa[s][0], 0u, qa[s][1], 0u};
        mma_16816_bf16(s0, qa4, kb[0], kb[1]);
        mma_16816_bf16(s1, qa4, kb[2], kb[3]);
      }
      const int tb = 2 * t4;
      float x[4] = {s0[0] * qs, s0[1] * qs, s1[0] * qs, s1[1] * qs};
      if (tb >= nv) x[0] = -INFINITY;
      if (tb + 1 >= nv) x[1] = -INFINITY;
      if (tb + 8 >= nv) x[2] = -INFINITY;
      if (tb + 9 >= nv) x[3] = -INFINITY;
      float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float mnew = fmaxf(m_run, tmax);  // finite: token 0 of a tile is live
      s_run = s_run * exp2f(m_run - mnew) + ((exp2f(x[0] - mnew) + exp2f(x[1] - mnew)) +
                                             (exp2f(x[2] - mnew) + exp2f(x[3] - mnew)));
      m_run = mnew;
    }
    __syncwarp();  // the stage is read before its next copy
    if (k % stp == stp - 1) {  // the page's last tile: its (m, s) per query head
      float s_tot = s_run + __shfl_xor_sync(0xffffffffu, s_run, 1);
      s_tot += __shfl_xor_sync(0xffffffffu, s_tot, 2);
      if (t4 == 0 && g < G) {
        float *dst = a.pm + (((size_t)unit * a.max_pages + tile_page(k)) * G + g) * 2;
        dst[0] = m_run;
        dst[1] = s_tot;
      }
      m_run = -INFINITY;
      s_run = 0.f;
    }
  }
}

// ---- per-unit normalisation, keys and nucleus size -----------------------------------------
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
  __shared__ unsigned long long redu[kCovThreads / 32];
  __shared__ unsigned long long hmass[kCovHist][256];  // warp w counts into copy w % kCovHist
  __shared__ int hcount[kCovHist][256];
  __shared__ unsigned long long scan_m[kCovThreads / 32];
  __shared__ int scan_n[kCovThreads / 32];
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
  const float2 *pm2 = reinterpret_cast<const float2 *>(a.pm) + (size_t)unit * a.max_pages * G;
  // the group's normalisers in one pass: per head an online (max, sum) over the pages' pairs,
  // combined over the block
  __shared__ float2 redp[kCovThreads / 32][G];
  float M[G], Zinv[G];
  {
    float mr[G], zr[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mr[g] = -INFINITY;
      zr[g] = 0.f;
    }
    auto fold = [](float &m, float &z, float mo, float zo) {  // (m, z) += (mo, zo), both relative to their max
      const float mn = fmaxf(m, mo);
      if (mn == -INFINITY) return;
      z = (m == -INFINITY ? 0.f : z * exp2f(m - mn)) + (mo == -INFINITY ? 0.f : zo * exp2f(mo - mn));
      m = mn;
    };
#pragma unroll 4
    for (int p = tid; p < P; p += kCovThreads)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 ms = pm2[(size_t)p * G + g];
        fold(mr[g], zr[g], ms.x, ms.y);
      }
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mo = __shfl_xor_sync(0xffffffffu, mr[g], o);
        const float zo = __shfl_xor_sync(0xffffffffu, zr[g], o);
        fold(mr[g], zr[g], mo, zo);
      }
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g) redp[warp][g] = make_float2(mr[g], zr[g]);
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float m = -INFINITY, z = 0.f;
#pragma unroll
      for (int w = 0; w < kCovThreads / 32; ++w) fold(m, z, redp[w][g].x, redp[w][g].y);
      M[g] = m;
      Zinv[g] = z > 0.f ? 1.f / z : 0.f;
    }
  }
  // page masses, keys, fixed-point masses
  uint32_t *krow = a.keys + (size_t)unit * a.key_stride;
  unsigned long long *qrow = a.qmass + (size_t)unit * a.max_pages;
  unsigned long long forced_q = 0, total_q = 0;
  int n_cand = 0;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;  // of the candidates' keys
#pragma unroll 4
  for (int p = tid; p < P; p += kCovThreads) {
    float mass = 0.f;
    bool read = false;  // false only for a page whose block id was out of range (flagged)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 ms = pm2[(size_t)p * G + g];
      if (ms.x != -INFINITY) {
        read = true;
        mass = fmaxf(mass, ms.y * exp2f(ms.x - M[g]) * Zinv[g]);
      }
    }
    const unsigned long long qm = (unsigned long long)((double)mass * kMassQuant + 0.5);
    if (a.masses_out) a.masses_out[(size_t)unit * a.max_pages + p] = mass;
    const bool forced = always_kept(p, P, a.sink, a.window);
    const uint32_t key = (forced || !read) ? 0u : score_key(mass);
    krow[p] = key;
    qrow[p] = qm;
    total_q += qm;
    if (forced) forced_q += qm;
    else if (read) ++n_cand;
    if (key != 0u) {
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
  total_q = block_sum_u64(total_q, redu);
  forced_q = block_sum_u64(forced_q, redu);
  n_cand = (int)block_sum_u64((unsigned long long)n_cand, redu);
  {  // the candidates' smallest and largest key over the block
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (lane == 0) {  // the scan arrays are not in use yet (redu may still be read)
      scan_n[warp] = (int)kmin;
      scan_m[warp] = kmax;
    }
    __syncthreads();
    kmin = 0xFFFFFFFFu;
    kmax = 0u;
#pragma unroll
    for (int w = 0; w < kCovThreads / 32; ++w) {
      kmin = min(kmin, (uint32_t)scan_n[w]);
      kmax = max(kmax, (uint32_t)scan_m[w]);
    }
  }
  __syncthreads();  // keys and masses of the row are written (each thread reads back any of them)
  const unsigned long long target = (unsigned long long)ceil((double)total_q * a.coverage);
  int k = 0;
  if (forced_q < target && n_cand > 0) {
    // MSB-first radix over the candidates' keys, starting at the highest bit where their
    // smallest and largest key differ (as the selection kernel does): per 8-bit digit a count
    // and a fixed-point mass histogram (kCovHist copies against atomic contention), then the
    // first digit, in descending order, whose running mass reaches what is still needed
    unsigned long long need = target - forced_q;  // mass still to cover
    int taken = 0;                                // keys above the running prefix
    const uint32_t diff = kmin ^ kmax;
    const int top = diff ? 31 - __clz(diff) : 0;
    int shift = top >= 7 ? top - 7 : 0;
    uint32_t prefix = shift + 8 >= 32 ? 0u : (kmin >> (shift + 8)) << (shift + 8);
    uint32_t mask = shift + 8 >= 32 ? 0u : (0xFFFFFFFFu << (shift + 8));
    const int lane = tid & 31, warp = tid >> 5;
    bool all = false;
#pragma unroll 1
    for (;;) {
      for (int x = tid; x < kCovHist * 256; x += kCovThreads) {
        (&hmass[0][0])[x] = 0ull;
        (&hcount[0][0])[x] = 0;
      }
      if (tid == 0) pick[0] = -1;
      __syncthreads();
#pragma unroll 4
      for (int p = tid; p < P; p += kCovThreads) {
        const uint32_t key = krow[p];
        if (key != 0u && (key & mask) == prefix) {
          const uint32_t bin = (key >> shift) & 255u;
          atomicAdd(&hmass[warp % kCovHist][bin], qrow[p]);
          atomicAdd(&hcount[warp % kCovHist][bin], 1);
        }
      }
      __syncthreads();
      // thread t owns digit 255 - t: descending digit order is thread order
      const int bin = 255 - tid;
      unsigned long long m = 0;
      int n = 0;
#pragma unroll
      for (int c = 0; c < kCovHist; ++c) {
        m += hmass[c][bin];
        n += hcount[c][bin];
      }
      unsigned long long incl_m = m;
      int incl_n = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long ym = __shfl_up_sync(0xffffffffu, incl_m, o);
        const int yn = __shfl_up_sync(0xffffffffu, incl_n, o);
        if (lane >= o) {
          incl_m += ym;
          incl_n += yn;
        }
      }
      if (lane == 31) {
        scan_m[warp] = incl_m;
        scan_n[warp] = incl_n;
      }
      __syncthreads();
      for (int w = 0; w < warp; ++w) {
        incl_m += scan_m[w];
        incl_n += scan_n[w];
      }
      const unsigned long long excl_m = incl_m - m;
      if (excl_m < need && incl_m >= need && n > 0) {  // exactly one digit qualifies, or none
        pick[0] = bin;
        pick[1] = incl_n - n;  // keys above this digit
        pick[2] = n;
        pick_mass[0] = excl_m;
        pick_mass[1] = m;
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
      if (shift == 0 || pick[2] == 1) {
        // every key equal to prefix has the same mass (a single key: it alone): how many of
        // them make up `need`
        const unsigned long long each = pick_mass[1] / (unsigned long long)pick[2];
        const unsigned long long n_eq = each > 0 ? (need + each - 1) / each : (unsigned long long)pick[2];
        taken += (int)min((unsigned long long)pick[2], max(1ull, n_eq));
        break;
      }
      shift = shift >= 8 ? shift - 8 : 0;  // an overlap with bits already fixed is harmless
      __syncthreads();                     // pick is rewritten by the next pass
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
  cudaError_t e = cudaErrorInvalidValue;
  bool done = false;
  if constexpr (sizeof(T) == 2) {
    if (tuning().decode_mma) {  // the tensor-core tiles of the decode, K only
      CUtensorMap tmK;
      if (!encode_cache_map(&tmK, c.k_cache, PSK_BF16, D, c.H_kv, (long long)c.nb * c.ps, 16, true))
        return cudaErrorInvalidValue;
      e = launch_kernel(true, page_mass_mma_kernel<D, G>, g1, kMassMmaWarps * 32, mass_mma_smem<D>(), s, c, tmK);
      done = true;
    }
  }
  if (!done) e = launch_kernel(true, page_mass_kernel<T, D, G>, g1, kMassThreads, 0, s, c);
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
