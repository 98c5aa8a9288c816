// Gaussian page score from the per-page key mean / std summaries (EntmaxKV README,
// introduction: pages are scored from per-page key statistics, "mean/std for Gaussian"; "Two
// selection strategies", Gaussian-aware: each page's scores modelled as a Gaussian, pages kept
// whose estimated maximum is high). For query head g and page p the logits q_g . k_t of the
// page's tokens are taken as Gaussian with mean q_g . mean_p and variance
// sum_d q_gd^2 std_pd^2 (dimensions independent); the page's estimated maximum is mean + z * std:
//
//   score[i,h,p] = scale * max_{g in group(h)} (q_g . mean_p + z * sqrt(sum_d (q_gd std_pd)^2)).
//
// gauss_score_kernel: one CTA of eight warps per (chunk of kGPages pages, sequence, group of up
// to 8 KV heads). The fp32 mean / std rows of a page for the group's heads are one contiguous
// run ([num_blocks, H_kv, 2, D]), so warp 0 fetches each page with one bulk copy (TMA engine)
// into a two-stage shared-memory ring, completion on one mbarrier per stage (bounded waits), as
// the bound's score kernel does. Warp w takes KV head w % hpc of the group (and every
// (8 / hpc)-th page of a stage); each lane reads its D/32 dims of the head's mean and std rows
// from shared memory, keeps q and q^2 of the G query heads for those dims in registers, and the
// G means and variances are reduced across the warp. The kernel writes the same selection keys as
// the bound's score kernel (0 for an always-kept page or a flagged block), and the selection
// kernel (select.cu) keeps the top-b. Without scores_out the always-kept pages' statistics are
// not read.
#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr int kGThreads = 256;
constexpr int kGWarps = kGThreads / 32;
constexpr int kGPages = 32;           // pages per CTA
constexpr int kGStages = 2;
constexpr int kGStageBytes = 32768;   // 4 pages of 8 heads x 2 x 128 fp32
constexpr int kGMaxStagePages = 32;

// Sums the NV values v[] over the 32 lanes with a transposing butterfly: each of the first
// log2(NV) steps (masks 16, 8, ...) hands the partner half of the values a lane carries, the
// rest are plain steps. On return v[0] holds, on every lane, the full sum of value index
// (lane >> (5 - log2 NV)) (lane bit 4 is that index's top bit).
template <int NV>
__device__ __forceinline__ void warp_transpose_sum(float (&v)[NV], int lane) {
  int L = NV;
#pragma unroll
  for (int mask = 16; mask >= 1; mask >>= 1) {
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

template <typename T, int D, int G>
__global__ void __launch_bounds__(kGThreads) gauss_score_kernel(ScoreArgs a, const float *stats, float z) {
  pdl_wait();  // the selection launch waits for this grid's completion
  constexpr int VPL = D / 32;  // dims per lane: 2 or 4
  static_assert(VPL == 2 || VPL == 4, "head_dim 64 or 128");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kGStages];
  __shared__ int okflag[kGStages][kGMaxStagePages];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hpc = a.H_kv < kGWarps ? a.H_kv : kGWarps;  // heads per CTA
  const int ngroups = a.H_kv / hpc;
  const int i = blockIdx.y / ngroups, h0 = (blockIdx.y - i * ngroups) * hpc;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by the selection kernel
  const int p0 = blockIdx.x * kGPages;
  if (p0 >= P) return;
  const int p1 = min(P, p0 + kGPages);
  const int page_bytes = hpc * 2 * D * 4;
  const int sp = min(kGMaxStagePages, kGStageBytes / page_bytes);
  const int n_stages = (p1 - p0 + sp - 1) / sp;
  const int32_t *bt = a.block_table + (size_t)i * a.max_pages;
  const int hh = warp % hpc, wg = warp / hpc, ng = kGWarps / hpc;
  const int h = h0 + hh;

  if (tid == 0) {
    for (int k = 0; k < kGStages; ++k) mbar_init(smem_u32(&bars[k]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t stream_policy = l2_evict_first_policy();
  auto produce = [&](int st) {  // warp 0: the pages of stage st into slot st % kGStages
    const int slot = st % kGStages;
    const int p = p0 + st * sp + lane;
    const bool in_chunk = lane < sp && p < p1;
    const int blk = in_chunk ? __ldg(bt + p) : -1;
    const bool valid = blk >= 0 && blk < a.nb;
    if (in_chunk && !valid) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    const bool needed = a.scores_out != nullptr || !always_kept(p, P, a.sink, a.window);
    const bool ok = in_chunk && valid && needed;
    if (lane < sp) okflag[slot][lane] = ok;
    const unsigned mask = __ballot_sync(0xffffffffu, ok);
    const uint32_t bar = smem_u32(&bars[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(mask) * page_bytes);
    __syncwarp();
    if (ok)
      bulk_g2s_stream(smem_u32(smem_raw + (size_t)slot * kGStageBytes + (size_t)lane * page_bytes),
                      stats + ((size_t)blk * a.H_kv + h0) * 2 * D, page_bytes, bar, stream_policy);
  };
  if (warp == 0)
    for (int st = 0; st < kGStages && st < n_stages; ++st) produce(st);

  // q and q^2 of the group's G query heads for this lane's dims, fp32
  float qv[G][VPL], q2[G][VPL];
  {
    const T *qrow = reinterpret_cast<const T *>(a.q) + ((size_t)i * a.H_q + (size_t)h * G) * D + lane * VPL;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < VPL; ++e) {
        float v;
        if constexpr (sizeof(T) == 2) {
          v = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(qrow)[(size_t)g * D + e] << 16);
        } else {
          v = reinterpret_cast<const float *>(qrow)[(size_t)g * D + e];
        }
        qv[g][e] = v;
        q2[g][e] = v * v;
      }
  }

  for (int st = 0; st < n_stages; ++st) {
    const int slot = st % kGStages;
    mbar_wait(smem_u32(&bars[slot]), (st / kGStages) & 1, a.ws);
    const int pb = p0 + st * sp;
    const int np = min(sp, p1 - pb);
    const unsigned char *stage = smem_raw + (size_t)slot * kGStageBytes;
    for (int j = wg; j < np; j += ng) {  // warp-uniform bound
      const float *row = reinterpret_cast<const float *>(stage + (size_t)j * page_bytes) + (size_t)hh * 2 * D + lane * VPL;
      float mu[VPL], var[VPL];
      if constexpr (VPL == 4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(row);
        const float4 s4 = *reinterpret_cast<const float4 *>(row + D);
        mu[0] = m4.x; mu[1] = m4.y; mu[2] = m4.z; mu[3] = m4.w;
        var[0] = s4.x * s4.x; var[1] = s4.y * s4.y; var[2] = s4.z * s4.z; var[3] = s4.w * s4.w;
      } else {
        const float2 m2 = *reinterpret_cast<const float2 *>(row);
        const float2 s2 = *reinterpret_cast<const float2 *>(row + D);
        mu[0] = m2.x; mu[1] = m2.y;
        var[0] = s2.x * s2.x; var[1] = s2.y * s2.y;
      }
      // the G means and G variances: value g is the mean of query head g, value G + g its
      // variance; after the transposing sum lane l holds value l >> (5 - log2 2G), so the
      // variance lanes are those with bit 4 set and their mean sits on lane ^ 16
      constexpr int NV = 2 * G;
      float val[NV];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float m = 0.f, v = 0.f;
#pragma unroll
        for (int e = 0; e < VPL; ++e) {
          m = fmaf(qv[g][e], mu[e], m);
          v = fmaf(q2[g][e], var[e], v);
        }
        val[g] = m;
        val[G + g] = v;
      }
      warp_transpose_sum<NV>(val, lane);
      const float mean_g = __shfl_xor_sync(0xffffffffu, val[0], 16);
      float best = fmaf(z, sqrtf(fmaxf(val[0], 0.f)), mean_g);  // meaningful on the variance lanes
      // max over the query heads: the variance lanes of different heads differ in bits 3 .. 5 - log2 2G
#pragma unroll
      for (int o = 8; o >= 16 / G; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
      if (lane == 16) {  // a variance lane holding the max over the group
        const int p = pb + j;
        const int unit = i * a.H_kv + h;
        const float sc = best * a.scale;
        const bool forced = always_kept(p, P, a.sink, a.window);
        a.keys[(size_t)unit * a.key_stride + p] = (okflag[slot][j] && !forced) ? score_key(sc) : 0u;
        if (a.scores_out) a.scores_out[(size_t)unit * a.max_pages + p] = sc;
      }
    }
    __syncthreads();  // every warp is done with this slot
    if (warp == 0 && st + kGStages < n_stages) {
      fence_proxy_async_smem();
      produce(st + kGStages);
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
  const int hpc = a.H_kv < kGWarps ? a.H_kv : kGWarps;
  if (a.H_kv % hpc != 0) return cudaErrorInvalidValue;
  const size_t smem = (size_t)kGStages * kGStageBytes;
  dim3 grid((a.max_pages + kGPages - 1) / kGPages, a.B * (a.H_kv / hpc));
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
