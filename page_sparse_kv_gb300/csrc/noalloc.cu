// psk_sparse_paged_decode_noalloc: the sparse decode for callers that cannot hand the library a
// workspace. Some hosts own all device memory themselves and give a plugin only its input and
// output buffers (a serving engine with its own pooled allocator and a fixed memory budget, or a
// real-time loop that must never enter cudaMalloc and its possible device synchronisation). For
// them the split-K partials live in a fixed, file-scope device array instead of a caller buffer.
//
// The array is kNoAllocScratchBytes (32 MiB) per GPU that loads it, held until the process
// exits. Problems whose partials do not fit are rejected with PSK_ERR_WORKSPACE. Only the GQA
// split decode is served (per-KV-head rows, values in device memory); latent caches return
// PSK_ERR_UNSUPPORTED.
//
// Host code cannot use the array's name as a device address (on the host it is only a stand-in
// symbol). Each call, with the caller's device current, looks the address up with
// cudaGetSymbolAddress in the current context, so a device reset or a context the caller made
// current through the driver API never leaves a stale address behind. With lazy module loading
// (the CUDA default) the first call on each device loads the module that holds the array, which
// may synchronise: make one warm-up call before any stream capture or latency-critical loop (or
// set CUDA_MODULE_LOADING=EAGER). Every call shares the one array and keeps the previous call's
// contents: the header (status word and merge tickets) is zeroed at the start of each call, and
// calls that overlap on the GPU (different streams, or different host threads) race on it and
// must be serialised by the caller. Device-side input violations are flagged in this internal
// header, which is not reported back; validate inputs with the workspace entry point if that
// matters.
//
// No counterpart exists in the pages this library follows.
#include "psk_common.cuh"
#include "psk_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_psk_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context.
int scratch_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_psk_noalloc_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();
    return PSK_ERR_CUDA;
  }
  *out = p;
  return PSK_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int psk_sparse_paged_decode_noalloc(const psk_layout *layout, const void *q, const void *k_cache,
                                               const void *v_cache, const int32_t *block_table,
                                               const int32_t *seq_lens, const int32_t *selected, int32_t b_max,
                                               float scale, void *out, psk_stream_t stream) {
  using namespace psk;
  if (!layout) return PSK_ERR_INVALID_ARG;
  const psk_layout &L = *layout;
  if (L.batch < 1 || L.num_q_heads < 1 || L.num_kv_heads < 1 || L.head_dim < 1 || L.v_head_dim < 1 ||
      L.page_size < 1 || L.num_blocks < 1 || L.max_pages < 1 || L.num_q_heads % L.num_kv_heads != 0 ||
      (L.dtype != PSK_F32 && L.dtype != PSK_BF16) || (L.latent != 0 && L.latent != 1))
    return PSK_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !selected || !out || b_max < 1)
    return PSK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PSK_ERR_INVALID_ARG;
  const int G = L.num_q_heads / L.num_kv_heads;
  if (L.latent || !decode_supported(L.dtype, L.head_dim, L.v_head_dim, G, L.page_size)) return PSK_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (!plan_decode(L, b_max, false, &plan)) return PSK_ERR_UNSUPPORTED;
  if (plan.ws_bytes > kNoAllocScratchBytes) return PSK_ERR_WORKSPACE;  // partials exceed the fixed scratch

  void *scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != PSK_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t units = (size_t)L.batch * L.num_kv_heads;
  if (cudaMemsetAsync(scratch, 0, ws_scratch_offset(units), s) != cudaSuccess) return PSK_ERR_CUDA;

  unsigned char *ws = static_cast<unsigned char *>(scratch);
  DecodeArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.selected = selected;
  a.out = out;
  a.ws = scratch;
  a.part_o = reinterpret_cast<float *>(ws + plan.off_o);
  a.part_ml = reinterpret_cast<float *>(ws + plan.off_ml);
  a.tickets = reinterpret_cast<uint32_t *>(ws + plan.off_tickets);
  a.B = L.batch;
  a.H_q = L.num_q_heads;
  a.H_kv = L.num_kv_heads;
  a.H_kv_cache = L.num_kv_heads;
  a.kv_shift = 0;
  a.v_host = 0;
  a.v_hot = nullptr;
  a.v_slot = nullptr;
  a.n_slots = 0;
  a.D = L.head_dim;
  a.D_v = L.v_head_dim;
  a.ps = L.page_size;
  a.nb = L.num_blocks;
  a.max_pages = L.max_pages;
  a.b_max = b_max;
  a.sw = plan.sw;
  a.n_items_max = plan.n_items_max;
  a.flat = plan.flat;
  a.taper = plan.taper;
  a.counts = reinterpret_cast<int32_t *>(ws + plan.off_counts);
  a.scale = scale;
  return launch_decode(a, L.dtype, s) == cudaSuccess ? PSK_OK : PSK_ERR_CUDA;
}
