// Device helpers shared by the psk kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <utility>

#include "../../include/psk.h"

namespace psk {

// ------------------------------------------------------------------------------------
// workspace header: the first 256 bytes of every workspace
// ------------------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;
struct WsHeader {
  uint32_t status;  // sticky PSK_DEV_* bits
};

__device__ __forceinline__ void set_status(void *ws, uint32_t bit) {
  atomicOr(&reinterpret_cast<WsHeader *>(ws)->status, bit);
}

// ------------------------------------------------------------------------------------
// Programmatic dependent launch: every kernel is launched with programmatic stream
// serialisation, so it may be scheduled while the kernel before it in the stream drains. Its
// first act is pdl_begin(): griddepcontrol.wait blocks until the previous grid has completed and
// its writes are visible (no global memory is touched before it, so any producer / consumer
// order, and any reuse of a buffer, is as safe as with plain stream order), then
// griddepcontrol.launch_dependents lets the next kernel in the stream be scheduled once every
// CTA of this grid has started. In a kernel launched without the attribute both are no-ops.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
  pdl_wait();
  pdl_trigger();
}

// Which launches carry the attribute: kernels that follow another kernel of the same call always
// (score after q split, select after score, flat decode after counts), the first kernel of a call
// too unless PSK_PDL=2; PSK_PDL=0 launches every kernel in plain stream order.
bool pdl_enabled(bool first_of_call);

// Host-side facts the launchers need, each computed once per device and cached (they never
// change for a device): its SM count, and per (kernel, threads, dynamic shared memory) the
// opt-in shared-memory limit set on the kernel and its resident CTAs per SM.
int sm_count();
// Sets the kernel's dynamic shared-memory limit to at least `smem` (once per device) and, when
// per_sm is given, returns its occupancy in CTAs per SM for `threads` threads.
cudaError_t kernel_setup(const void *fn, int threads, size_t smem, int *per_sm = nullptr);
// Drops the cached set-up of a kernel on the current device (after a launch failed, e.g. because
// a device reset discarded the attribute), so the next kernel_setup sets it again.
void kernel_forget(const void *fn);

// Tuning overrides from the environment, read once per process: PSK_SCORE_TAIL (pages),
// PSK_SCORE_TAIL_CHUNK, PSK_SCORE_PCHUNK, PSK_SELECT_CHUNK (pages per selection CTA: 1024, 2048,
// 4096, 8192 or 16384; raised while the chunks' candidates exceed the merge), PSK_SCORE_MMA (0: bf16 page scores on the FMA pipe
// instead of the tensor cores), PSK_DECODE_MMA (0: bf16 decode tiles on the FMA pipe),
// PSK_DECODE_LAYOUT ("split" / "flat"), PSK_DECODE_SPLIT (list entries per CTA),
// PSK_DECODE_NO_TAPER. -1 / 0 = not set.
struct Tuning {
  long long score_tail = -1;
  int score_tail_chunk = -1, score_pchunk = -1;
  int select_chunk = -1;
  bool score_mma = true;
  bool decode_mma = true;
  int decode_layout = 0;  // 0 default, 1 split, 2 flat
  int decode_split = -1;
  bool decode_no_taper = false;
};
const Tuning &tuning();

// Launch with the programmatic-serialisation attribute (when enabled for this kind of launch).
// The kernel's shared-memory limit is set (once per device, cached) before the launch; a launch
// that fails drops that cache entry and is tried once more after setting it again.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool first_of_call, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, const Args &...args) {
  const void *fn = reinterpret_cast<const void *>(kernel);
  cudaError_t e = kernel_setup(fn, (int)(block.x * block.y * block.z), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled(first_of_call) ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    kernel_forget(fn);
    if (kernel_setup(fn, (int)(block.x * block.y * block.z), smem) == cudaSuccess)
      e = cudaLaunchKernelEx(&cfg, kernel, args...);
  }
  return e;
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout shared by every call, so one buffer can serve all of them in stream order:
//   [0, 256)                      header (status word)
//   [256, 256 + 4 * units)        score/select merge tickets, one per (sequence, KV head)
//   [.., + 4 * units)             decode merge tickets
//   [ws_scratch_offset(units), ..) per-call scratch (candidates, split partials), which any
//                                 later call may overwrite
// Tickets are only ever touched by their own op and are back at zero when each call ends.
inline size_t ws_score_tickets_offset() { return kWsHeader; }
inline size_t ws_decode_tickets_offset(size_t units) { return kWsHeader + units * 4; }
inline size_t ws_scratch_offset(size_t units) { return align_up(kWsHeader + 2 * units * 4, 256); }

// ------------------------------------------------------------------------------------
// storage types: bf16 is carried as its 16-bit pattern
// ------------------------------------------------------------------------------------
struct bf16_t {
  uint16_t bits;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t *>(&b);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr int kPerChunk = 4;  // elements per 16-byte chunk
  __device__ __forceinline__ static void to_f2(const uint4 &c, float2 *out) {
    out[0] = make_float2(__uint_as_float(c.x), __uint_as_float(c.y));
    out[1] = make_float2(__uint_as_float(c.z), __uint_as_float(c.w));
  }
  // 8-byte group (2 elements) -> floats
  __device__ __forceinline__ static void to_f2_8(const uint2 &c, float2 *out) {
    out[0] = make_float2(__uint_as_float(c.x), __uint_as_float(c.y));
  }
  __device__ __forceinline__ static void store(float *p, float v) { *p = v; }
};
template <> struct Elem<bf16_t> {
  static constexpr int kBytes = 2;
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void to_f2(const uint4 &c, float2 *out) {
    out[0] = bf16x2_to_f2(c.x);
    out[1] = bf16x2_to_f2(c.y);
    out[2] = bf16x2_to_f2(c.z);
    out[3] = bf16x2_to_f2(c.w);
  }
  // 8-byte group (4 elements) -> floats
  __device__ __forceinline__ static void to_f2_8(const uint2 &c, float2 *out) {
    out[0] = bf16x2_to_f2(c.x);
    out[1] = bf16x2_to_f2(c.y);
  }
  __device__ __forceinline__ static void store(bf16_t *p, float v) { p->bits = f32_to_bf16_bits(v); }
};

// ------------------------------------------------------------------------------------
// order-preserving integer images
// ------------------------------------------------------------------------------------
// Signed-integer image of a float bit pattern under IEEE totalOrder (non-NaN):
// -0.0 sorts below +0.0, larger value -> larger integer.
__device__ __forceinline__ int32_t f32_order_key(uint32_t bits) {
  int32_t i = static_cast<int32_t>(bits);
  return i ^ ((i >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ int32_t bf16_order_key(uint32_t bits16) {
  int32_t i = static_cast<int32_t>(static_cast<int16_t>(static_cast<uint16_t>(bits16)));
  return i ^ ((i >> 15) & 0x7FFF);
}

// Unsigned selection key of a score: larger score -> larger key; -0.0 and +0.0 map to the
// same key (they tie). Key 0 is never produced by a finite score and marks "no candidate".
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------------------------
// packed fp32x2 FMA (sm_100+): d = a * b + c on both lanes
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ------------------------------------------------------------------------------------
// cp.async (16-byte, L2-only) with zero fill
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// copies 16 bytes when `pred`, else writes 16 zero bytes without reading global memory
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------------------------
// mbarrier + bulk (TMA engine) copies
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// Bounded wait for the phase with parity `parity`: gives up after `limit` polls (each poll may
// suspend the thread for a short hardware-defined time), sets PSK_DEV_TIMEOUT and returns false,
// so a lost copy can never hang the GPU. Every kernel waits with kMbarSpinLimit polls; the
// self-test entry point runs the same wait with a short limit on a phase that cannot complete.
constexpr uint32_t kMbarSpinLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, void *ws, uint32_t limit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  set_status(ws, PSK_DEV_TIMEOUT);
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, void *ws) {
  return mbar_wait_limit(bar, parity, ws, kMbarSpinLimit);
}
// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16), completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// L2 policy for data streamed once: evicted first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache-eviction policy.
__device__ __forceinline__ void bulk_g2s_stream(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar), "l"(pol)
               : "memory");
}

// 3-D tiled tensor copy global -> shared (TMA), completing on `bar`. The innermost coordinate
// is always 0 here, so it meets the 16-byte start rule for every element type.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// tma_load_3d with an L2 cache-eviction policy.
__device__ __forceinline__ void tma_load_3d_stream(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar,
                                                   uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

// Host: encode a 3-D tiled tensor map over a paged cache [rows, H, D] (elements of `dtype`) with
// a box of `box_rows` rows x 1 head x D elements, or, with sw128, x 128 bytes of elements stored
// with the 128-byte swizzle (a row then takes D * size / 128 boxes). Returns false on failure.
bool encode_cache_map(CUtensorMap *map, const void *base, int dtype, int D, int H, long long rows, int box_rows,
                      bool sw128 = false);
// Host: 2-D bf16 tensor map over a row-major [rows, cols] matrix with a {box_cols, box_rows}
// box and the 128-byte swizzle (box_cols * 2 must be 128).
bool encode_matrix_map_sw128(CUtensorMap *map, const void *base, long long cols, long long rows, int box_cols,
                             int box_rows);

// 2-D tiled tensor copy global -> shared (TMA); x * 2 bytes must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------------------------
// warp-level tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate) and its operand loads
// ------------------------------------------------------------------------------------
// Four 8x8 b16 matrices from shared memory: lanes 8j .. 8j + 7 give the 16-byte row addresses of
// matrix j, which lands in r[j] (row lane / 4, elements 2 (lane % 4) and + 1).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// The same, transposed: r[j] holds rows 2 (lane % 4) and + 1 of column lane / 4 of matrix j.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// c += A (16 x 16, row-major fragment) * B (16 x 8, column-major fragment), fp32 accumulate.
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two fp32 values rounded to bf16 (nearest even) in one word: lo in bits 0..15, hi in 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace psk
