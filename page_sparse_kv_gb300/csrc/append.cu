// Stage 1: write appended tokens into the paged cache and refresh the per-page, per-KV-head
// elementwise key min / max summaries (EntmaxKV README, kernels/page_metadata.py "per-page
// k_min / k_max refresh"; the decode call appends k_new / v_new before scoring) and, when asked,
// the per-page key mean / std summaries (EntmaxKV README, introduction, "mean/std for
// Gaussian"; gaussian/page_metadata.py "Per-page k_mean / k_std refresh").
//
// One CTA per (sequence, touched page). Each thread owns one 16-byte chunk of a token row
// (H_kv * D elements) and walks the page's new tokens: it copies the chunk into the cache
// and folds it into a running min / max in registers, then writes the chunk's summary
// once. A page that already held tokens before start_pos starts from its stored summary;
// a page whose first token is new starts fresh. min / max use the totalOrder integer image
// of the bit pattern, so -0.0 < +0.0 and the result is bit-exact in any storage dtype.
#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

template <typename T> struct MinMax;

template <> struct MinMax<bf16_t> {
  __device__ __forceinline__ static uint32_t lo16(uint32_t a, uint32_t b) {
    return bf16_order_key(a & 0xFFFF) <= bf16_order_key(b & 0xFFFF) ? (a & 0xFFFF) : (b & 0xFFFF);
  }
  __device__ __forceinline__ static uint32_t hi16(uint32_t a, uint32_t b) {
    return bf16_order_key(a & 0xFFFF) >= bf16_order_key(b & 0xFFFF) ? (a & 0xFFFF) : (b & 0xFFFF);
  }
  __device__ __forceinline__ static uint32_t lo_word(uint32_t a, uint32_t b) {
    return lo16(a, b) | (lo16(a >> 16, b >> 16) << 16);
  }
  __device__ __forceinline__ static uint32_t hi_word(uint32_t a, uint32_t b) {
    return hi16(a, b) | (hi16(a >> 16, b >> 16) << 16);
  }
};
template <> struct MinMax<float> {
  __device__ __forceinline__ static uint32_t lo_word(uint32_t a, uint32_t b) {
    return f32_order_key(a) <= f32_order_key(b) ? a : b;
  }
  __device__ __forceinline__ static uint32_t hi_word(uint32_t a, uint32_t b) {
    return f32_order_key(a) >= f32_order_key(b) ? a : b;
  }
};

template <typename T>
__device__ __forceinline__ uint4 chunk_min(uint4 a, uint4 b) {
  return make_uint4(MinMax<T>::lo_word(a.x, b.x), MinMax<T>::lo_word(a.y, b.y), MinMax<T>::lo_word(a.z, b.z),
                    MinMax<T>::lo_word(a.w, b.w));
}
template <typename T>
__device__ __forceinline__ uint4 chunk_max(uint4 a, uint4 b) {
  return make_uint4(MinMax<T>::hi_word(a.x, b.x), MinMax<T>::hi_word(a.y, b.y), MinMax<T>::hi_word(a.z, b.z),
                    MinMax<T>::hi_word(a.w, b.w));
}

// Mean and population standard deviation of the page's valid tokens [0, n_valid) for the
// elements of chunk c (one KV head's EPC consecutive dims), in fp32 by two passes over the
// cache rows, written to stats. The rows this thread wrote in this launch are its own chunk's, so
// program order makes them visible to it.
template <typename T>
__device__ __forceinline__ void refresh_page_stats(const AppendArgs &a, int blk, int n_valid, int c) {
  constexpr int EPC = Elem<T>::kPerChunk;
  const int cpr_k = a.D / EPC;
  const int h = c / cpr_k;
  const int e0 = (c - h * cpr_k) * EPC;
  const size_t row_k = (size_t)a.H_kv * a.D;
  const T *kc = reinterpret_cast<const T *>(a.k_cache) + (size_t)blk * a.ps * row_k + (size_t)c * EPC;
  float sum[EPC];
#pragma unroll
  for (int e = 0; e < EPC; ++e) sum[e] = 0.f;
  for (int r = 0; r < n_valid; ++r) {
    float2 f[EPC / 2];
    Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(kc + (size_t)r * row_k), f);
#pragma unroll
    for (int e = 0; e < EPC / 2; ++e) {
      sum[2 * e] += f[e].x;
      sum[2 * e + 1] += f[e].y;
    }
  }
  const float inv_n = 1.f / (float)n_valid;
  float mean[EPC], m2[EPC];
#pragma unroll
  for (int e = 0; e < EPC; ++e) {
    mean[e] = sum[e] * inv_n;
    m2[e] = 0.f;
  }
  for (int r = 0; r < n_valid; ++r) {
    float2 f[EPC / 2];
    Elem<T>::to_f2(*reinterpret_cast<const uint4 *>(kc + (size_t)r * row_k), f);
#pragma unroll
    for (int e = 0; e < EPC / 2; ++e) {
      const float d0 = f[e].x - mean[2 * e], d1 = f[e].y - mean[2 * e + 1];
      m2[2 * e] = fmaf(d0, d0, m2[2 * e]);
      m2[2 * e + 1] = fmaf(d1, d1, m2[2 * e + 1]);
    }
  }
  float *dst = a.stats + ((size_t)blk * a.H_kv + h) * 2 * a.D + e0;
#pragma unroll
  for (int e = 0; e < EPC; ++e) {
    dst[e] = mean[e];
    dst[a.D + e] = sqrtf(m2[e] * inv_n);
  }
}

template <typename T>
__global__ void append_summarize_kernel(AppendArgs a) {
  pdl_begin();
  const int i = blockIdx.y;
  const int j = blockIdx.x;
  const int c0 = a.cu_new[i];
  const int n = a.cu_new[i + 1] - c0;
  const int s0 = a.start_pos[i];
  if (n <= 0 || s0 < 0) {
    if ((n < 0 || s0 < 0) && j == 0 && threadIdx.x == 0) set_status(a.ws, PSK_DEV_BAD_APPEND);
    return;
  }
  const int ps = a.ps;
  const int p = s0 / ps + j;
  const int last = (s0 + n - 1) / ps;
  if (p > last) return;
  if (p >= a.max_pages) {
    if (threadIdx.x == 0) set_status(a.ws, PSK_DEV_BAD_APPEND);
    return;
  }
  const int blk = a.block_table[(size_t)i * a.max_pages + p];
  if (blk < 0 || blk >= a.nb) {
    if (threadIdx.x == 0) set_status(a.ws, PSK_DEV_BAD_BLOCK);
    return;
  }
  const int t_lo = max(p * ps, s0);
  const int t_hi = min((p + 1) * ps, s0 + n);
  const bool fresh = p * ps >= s0;  // no token of this page predates the call

  constexpr int EPC = Elem<T>::kPerChunk;
  const int cpr_k = a.D / EPC;                // chunks per head row of K
  const int nck = a.H_kv * cpr_k;             // chunks per token row of K
  const size_t row_k = (size_t)a.H_kv * a.D;  // elements per token row
  const T *kn = reinterpret_cast<const T *>(a.k_new);
  T *kc = reinterpret_cast<T *>(a.k_cache);
  T *sm = reinterpret_cast<T *>(a.summaries);

  const int ncv = a.v_cache ? a.H_kv * (a.D_v / EPC) : 0;  // latent cache: the value is part of the key row
  const size_t row_v = (size_t)a.H_kv * a.D_v;
  const T *vn = reinterpret_cast<const T *>(a.v_new);
  T *vc = reinterpret_cast<T *>(a.v_cache);
  if (t_hi - t_lo == 1 && nck <= (int)blockDim.x && ncv <= (int)blockDim.x) {
    // one new token on this page (the decode step): every load of the thread is issued before
    // any store, so the page costs one round trip after its block id
    const int c = threadIdx.x;
    const int t = t_lo;
    uint4 x{}, olo{}, ohi{}, xv{};
    T *sum_lo = nullptr;
    if (c < nck) {
      const int h = c / cpr_k;
      const int e0 = (c - h * cpr_k) * EPC;
      if (sm) sum_lo = sm + ((size_t)blk * a.H_kv + h) * 2 * a.D + e0;
      x = __ldg(reinterpret_cast<const uint4 *>(kn + (size_t)(c0 + t - s0) * row_k + (size_t)c * EPC));
      if (!fresh && sm) {
        olo = *reinterpret_cast<const uint4 *>(sum_lo);
        ohi = *reinterpret_cast<const uint4 *>(sum_lo + a.D);
      }
    }
    if (c < ncv) xv = __ldg(reinterpret_cast<const uint4 *>(vn + (size_t)(c0 + t - s0) * row_v + (size_t)c * EPC));
    if (c < nck) {
      *reinterpret_cast<uint4 *>(kc + ((size_t)blk * ps + (t - p * ps)) * row_k + (size_t)c * EPC) = x;
      if (sm) {
        *reinterpret_cast<uint4 *>(sum_lo) = fresh ? x : chunk_min<T>(olo, x);
        *reinterpret_cast<uint4 *>(sum_lo + a.D) = fresh ? x : chunk_max<T>(ohi, x);
      }
    }
    if (c < ncv) *reinterpret_cast<uint4 *>(vc + ((size_t)blk * ps + (t - p * ps)) * row_v + (size_t)c * EPC) = xv;
    if (a.stats && c < nck) refresh_page_stats<T>(a, blk, t_hi - p * ps, c);
    return;
  }

  for (int c = threadIdx.x; c < nck; c += blockDim.x) {
    const int h = c / cpr_k;
    const int e0 = (c - h * cpr_k) * EPC;
    T *sum_lo = sm ? sm + ((size_t)blk * a.H_kv + h) * 2 * a.D + e0 : nullptr;
    T *sum_hi = sm ? sum_lo + a.D : nullptr;
    uint4 lo, hi;
    int t = t_lo;
    const uint4 first = *reinterpret_cast<const uint4 *>(kn + (size_t)(c0 + t - s0) * row_k + (size_t)c * EPC);
    *reinterpret_cast<uint4 *>(kc + ((size_t)blk * ps + (t - p * ps)) * row_k + (size_t)c * EPC) = first;
    if (fresh || !sm) {
      lo = first;
      hi = first;
    } else {
      lo = chunk_min<T>(*reinterpret_cast<const uint4 *>(sum_lo), first);
      hi = chunk_max<T>(*reinterpret_cast<const uint4 *>(sum_hi), first);
    }
    for (++t; t < t_hi; ++t) {
      const uint4 x = *reinterpret_cast<const uint4 *>(kn + (size_t)(c0 + t - s0) * row_k + (size_t)c * EPC);
      *reinterpret_cast<uint4 *>(kc + ((size_t)blk * ps + (t - p * ps)) * row_k + (size_t)c * EPC) = x;
      lo = chunk_min<T>(lo, x);
      hi = chunk_max<T>(hi, x);
    }
    if (sm) {
      *reinterpret_cast<uint4 *>(sum_lo) = lo;
      *reinterpret_cast<uint4 *>(sum_hi) = hi;
    }
    if (a.stats) refresh_page_stats<T>(a, blk, t_hi - p * ps, c);
  }

  for (int c = threadIdx.x; c < ncv; c += blockDim.x) {
    for (int t = t_lo; t < t_hi; ++t) {
      const uint4 x = *reinterpret_cast<const uint4 *>(vn + (size_t)(c0 + t - s0) * row_v + (size_t)c * EPC);
      *reinterpret_cast<uint4 *>(vc + ((size_t)blk * ps + (t - p * ps)) * row_v + (size_t)c * EPC) = x;
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, int dtype, int max_new, cudaStream_t s) {
  const int es = dtype == PSK_F32 ? 4 : 2;
  const int chunks = max(a.H_kv * a.D * es / 16, a.v_cache ? a.H_kv * a.D_v * es / 16 : 0);
  const int threads = min(256, ((chunks + 31) / 32) * 32);
  const int pages = (max_new + a.ps - 2) / a.ps + 1;
  dim3 grid(pages, a.B);
  if (dtype == PSK_F32)
    return launch_kernel(true, append_summarize_kernel<float>, grid, threads, 0, s, a);
  else
    return launch_kernel(true, append_summarize_kernel<bf16_t>, grid, threads, 0, s, a);
}

}  // namespace psk
