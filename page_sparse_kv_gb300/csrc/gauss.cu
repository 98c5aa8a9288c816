// Gaussian page score from the per-page key mean / std summaries (EntmaxKV README,
// introduction: pages are scored from per-page key statistics, "mean/std for Gaussian"; "Two
// selection strategies", Gaussian-aware: each page's scores modelled as a Gaussian, pages kept
// whose estimated maximum is high). For query head g and page p the logits q_g . k_t of the
// page's tokens are taken as Gaussian with mean q_g . mean_p and variance
// sum_d q_gd^2 std_pd^2 (dimensions independent); the page's estimated maximum is mean + z * std:
//
//   score[i,h,p] = scale * max_{g in group(h)} (q_g . mean_p + z * sqrt(sum_d (q_gd std_pd)^2)).
//
// gauss_score_kernel: one CTA of eight warps per (chunk of 32 pages, sequence); warp w takes the
// (page, KV head) pairs w, w + 8, ... of the chunk; a pair's mean and std rows (fp32, D each)
// are read by the 32 lanes with one vector load each, and the G query heads' sums are reduced
// across the warp. The sequence's queries sit in shared memory as fp32. The kernel writes the
// same selection keys as the bound's score kernel (0 for an always-kept page or a flagged
// block), and the selection kernel (select.cu) keeps the top-b.
#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr int kGThreads = 256;
constexpr int kGPages = 32;

template <typename T, int D, int G>
__global__ void __launch_bounds__(kGThreads) gauss_score_kernel(ScoreArgs a, const float *stats, float z) {
  pdl_wait();  // the selection launch waits for this grid's completion
  constexpr int VPL = D / 32;  // dims per lane: 2 or 4
  static_assert(VPL == 2 || VPL == 4, "head_dim 64 or 128");
  extern __shared__ float qs_all[];  // [H_q][D] fp32
  const int i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by the selection kernel
  const int p0 = blockIdx.x * kGPages;
  if (p0 >= P) return;
  const int p1 = min(P, p0 + kGPages);
  const T *qrow = reinterpret_cast<const T *>(a.q) + (size_t)i * a.H_q * D;
  for (int x = tid; x < a.H_q * D; x += kGThreads) {
    float v;
    if constexpr (sizeof(T) == 2) {
      v = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(qrow)[x] << 16);
    } else {
      v = reinterpret_cast<const float *>(qrow)[x];
    }
    qs_all[x] = v;
  }
  __syncthreads();
  const int n_pairs = (p1 - p0) * a.H_kv;
  for (int x = warp; x < n_pairs; x += kGThreads / 32) {
    const int p = p0 + x / a.H_kv, h = x % a.H_kv;
    const int unit = i * a.H_kv + h;
    const int blk = a.block_table[(size_t)i * a.max_pages + p];
    const bool ok = blk >= 0 && blk < a.nb;
    if (!ok && lane == 0) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    float mu[VPL], sd[VPL];
    if (ok) {
      const float *row = stats + ((size_t)blk * a.H_kv + h) * 2 * D + lane * VPL;
      if constexpr (VPL == 4) {
        const float4 m4 = __ldcs(reinterpret_cast<const float4 *>(row));
        const float4 s4 = __ldcs(reinterpret_cast<const float4 *>(row + D));
        mu[0] = m4.x; mu[1] = m4.y; mu[2] = m4.z; mu[3] = m4.w;
        sd[0] = s4.x; sd[1] = s4.y; sd[2] = s4.z; sd[3] = s4.w;
      } else {
        const float2 m2 = __ldcs(reinterpret_cast<const float2 *>(row));
        const float2 s2 = __ldcs(reinterpret_cast<const float2 *>(row + D));
        mu[0] = m2.x; mu[1] = m2.y;
        sd[0] = s2.x; sd[1] = s2.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < VPL; ++e) mu[e] = sd[e] = 0.f;
    }
    float best = -INFINITY;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float *qg = qs_all + (size_t)(h * G + g) * D + lane * VPL;
      float m = 0.f, v = 0.f;
#pragma unroll
      for (int e = 0; e < VPL; ++e) {
        m = fmaf(qg[e], mu[e], m);
        const float t = qg[e] * sd[e];
        v = fmaf(t, t, v);
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        m += __shfl_xor_sync(0xffffffffu, m, o);
        v += __shfl_xor_sync(0xffffffffu, v, o);
      }
      best = fmaxf(best, fmaf(z, sqrtf(v), m));
    }
    if (lane == 0) {
      const float sc = best * a.scale;
      const bool forced = always_kept(p, P, a.sink, a.window);
      a.keys[(size_t)unit * a.key_stride + p] = (ok && !forced) ? score_key(sc) : 0u;
      if (a.scores_out) a.scores_out[(size_t)unit * a.max_pages + p] = sc;
    }
  }
}

}  // namespace

#define PSK_GAUSS_CASES(X)     \
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

bool gauss_supported(int dtype, int D, int G) {
#define X(TT, DT, DD, GG) \
  if (dtype == DT && D == DD && G == GG) return true;
  PSK_GAUSS_CASES(X)
#undef X
  return false;
}

cudaError_t launch_gauss_score_select(const ScoreArgs &a, const float *stats, float z, int dtype, cudaStream_t s) {
  const int D = a.D, G = a.H_q / a.H_kv;
  const size_t smem = (size_t)a.H_q * D * 4;
  dim3 grid((a.max_pages + kGPages - 1) / kGPages, a.B);
  cudaError_t e = cudaErrorInvalidValue;
#define X(TT, DT, DD, GG)                                                                                   \
  if (dtype == DT && D == DD && G == GG)                                                                    \
    e = launch_kernel(true, gauss_score_kernel<TT, DD, GG>, grid, kGThreads, smem, s, a, stats, z);
  PSK_GAUSS_CASES(X)
#undef X
  if (e != cudaSuccess) return e;
  return launch_page_select(a, s);
}

}  // namespace psk
