// The latent (MLA) form of the page score and the decode, on the 5th-generation tensor cores.
//
// 128 query heads share one latent KV head of 576 dims (the value is its first 512 dims), so
// both the Quest-style page bound and the attention are dense tile products here (LOCKS
// PKG-INFO, "How it works", MLA: the same page selection on the latent cache, max-unioned
// over the query heads; EntmaxKV README, Top-k: the Quest-style bound).
//
// Score: with qn = min(q, 0) and qp = max(q, 0) (exact in bf16), a page's bound for query head
// g is sum_d qn[g,d] * kmin[d] + qp[g,d] * kmax[d], i.e. the product of the page's summary row
// [kmin | kmax] (1152 elements, its stored layout) with [qn | qp]. One CTA computes
//   S^T[page, head] = Summ[128 pages x 1152] * Qs[128 heads x 1152]^T
// with tcgen05.mma (bf16 inputs, fp32 accumulation in tensor memory): M = 128 pages are the
// tensor-memory lanes and N = 128 heads the columns, so the max over the group is a loop over
// one thread's columns. Operands are staged per 64-element K block by cp.async with the
// 128-byte swizzle into a 3-stage ring; tcgen05.commit on a per-stage mbarrier frees a stage.
//
// Decode: one CTA per (split of the page list, half of the value dims, sequence). O for 128
// heads x 256 value dims fills 256 of the 512 tensor-memory columns, hence the split of D_v
// across two CTAs (each computes S itself). Q dims 0..383 live in tensor memory as the A
// operand of S = Q K^T (192 columns), dims 384..575 in shared memory (TMA, 128-byte swizzle);
// K tiles of 64 tokens x 576 (two 32-row TMA boxes per 64-dim block) stream through a 2-stage
// ring in two parts with their own full / empty mbarriers. Per tile: S (M = 128 heads, N = 64
// tokens) into tensor memory; each softmax thread owns one head's row: online softmax in fp32
// (log2 domain, lazy rescale), P written as bf16 to shared memory (128-byte swizzle); O += P V
// (N = 256 value dims, V read MN-major straight out of the K tile) accumulates in tensor
// memory. Six warps: four softmax warps (one thread per head), one warp whose lane 0 issues the
// MMAs (S of the next tile ahead of P.V of this one) and one whose lane 0 issues the TMA copies.
// Splits are merged by log-sum-exp: with at most 8 splits per (sequence, half) they run as one
// thread-block cluster, park their O rows and (m, l) in shared memory and each merge a slice of
// the value dims over distributed shared memory; with more, the last CTA of each (sequence,
// half) merges them from the workspace.
#include <algorithm>
#include <cstdlib>

#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

constexpr int kD = 576, kDv = 512, kHeads = 128;
constexpr int kKB = kD / 64;  // 64-element K blocks of a latent row
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------------------
// tcgen05 helpers
// ------------------------------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading / stride byte offsets, layout
// (2 = 128-byte swizzle, 4 = 64-byte swizzle), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7) << 61;
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K-major or
// MN-major, N and M.
__device__ __forceinline__ uint32_t umma_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// The same with A read from tensor memory (a_tmem: lane 0, first column of the K step; M = 128
// rows on the 128 lanes, two bf16 per 32-bit column).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%"
      "22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// 32 columns of this warp's 32 lanes; tmem_st32 waits for the store, tmem_st32_async does not
// (tmem_wait_st then waits for every store this thread issued)
__device__ __forceinline__ void tmem_st32_async(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%"
      "21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%"
      "21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
// thread-block cluster: this CTA's rank and the cluster's size (1 and 1 without a cluster launch),
// a shared-memory address of the same variable in CTA `rank`, loads through it, and the
// cluster-wide barrier (every thread of every CTA of the cluster, warp-converged)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// (a shared::cta address is also the shared::cluster address of this CTA's own shared memory)
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// ------------------------------------------------------------------------------------
// score
// ------------------------------------------------------------------------------------
// q [B, 128, 576] -> [B, 128, 1152] = [min(q, 0) | max(q, 0)] (bit operations on bf16: a
// negative value (sign set, -0.0 included) goes to the first half, the rest to the second).
__global__ void mla_qsplit_kernel(const uint16_t *q, uint16_t *qs, int rows) {
  pdl_begin();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * (kD / 8)) return;
  const int row = idx / (kD / 8), c = idx - row * (kD / 8);
  const uint4 w = *reinterpret_cast<const uint4 *>(q + (size_t)row * kD + c * 8);
  auto neg_mask = [](uint32_t x) { return ((x & 0x80008000u) >> 15) * 0xFFFFu; };
  const uint4 m = make_uint4(neg_mask(w.x), neg_mask(w.y), neg_mask(w.z), neg_mask(w.w));
  *reinterpret_cast<uint4 *>(qs + (size_t)row * 2 * kD + c * 8) = make_uint4(w.x & m.x, w.y & m.y, w.z & m.z, w.w & m.w);
  *reinterpret_cast<uint4 *>(qs + (size_t)row * 2 * kD + kD + c * 8) =
      make_uint4(w.x & ~m.x, w.y & ~m.y, w.z & ~m.z, w.w & ~m.w);
}

constexpr int kScStages = 3;
constexpr int kScStage = 32768;  // 16 KB of page rows + 16 KB of head rows (one 64-element K block each)
constexpr int kScSmem = 1024 + kScStages * kScStage;
constexpr int kScKBlocks = 2 * kD / 64;  // 18

__global__ void __launch_bounds__(128) mla_score_kernel(ScoreArgs a, const uint16_t *qs) {
  pdl_wait();  // dependents are released when this grid completes
  extern __shared__ unsigned char dyn[];
  unsigned char *base = align1024(dyn);
  __shared__ __align__(8) uint64_t bars[kScStages];
  __shared__ uint32_t tslot;
  const int i = blockIdx.y, tile = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  if (seq_len < 1 || P > a.max_pages) return;  // reported by the select kernel
  const int p0 = tile * 128;
  if (p0 >= P) return;
  // block id of every page row of the tile (0 and not loaded for rows past P or a bad block)
  __shared__ int row_blk[128];
  {
    const int p = p0 + tid;
    int blk = -1;
    if (p < P) {
      blk = a.block_table[(size_t)i * a.max_pages + p];
      if (blk < 0 || blk >= a.nb) {
        set_status(a.ws, PSK_DEV_BAD_BLOCK);
        blk = -1;
      }
      // always-kept pages are kept whatever their score: not read unless scores are requested
      if (!a.scores_out && always_kept(p, P, a.sink, a.window)) blk = -1;
    }
    row_blk[tid] = blk;
  }

  if (tid == 0) {
    for (int k = 0; k < kScStages; ++k) mbar_init(smem_u32(&bars[k]), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const uint16_t *qbase = qs + (size_t)i * kHeads * 2 * kD;
  const uint16_t *sbase = reinterpret_cast<const uint16_t *>(a.summaries);

  // One 64-element K block of 128 page rows and 128 head rows, 128-byte swizzle. Eight
  // consecutive threads copy the eight 16-byte chunks of one row, so every request of a warp
  // covers whole 128-byte lines.
  auto fill = [&](int kb, int st) {
    const uint32_t sa = smem_u32(base + st * kScStage), sb = sa + 16384;
    const int c = tid & 7;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = (tid >> 3) + 16 * k;
      const uint32_t off = r * 128 + ((c ^ (r & 7)) * 16);
      const int blk = row_blk[r];
      cp_async16(sa + off, sbase + (size_t)(blk < 0 ? 0 : blk) * 2 * kD + kb * 64 + c * 8, blk >= 0);
      cp_async16(sb + off, qbase + (size_t)r * 2 * kD + kb * 64 + c * 8, true);
    }
  };
  fill(0, 0);
  cp_async_commit();
  fill(1, 1);
  cp_async_commit();
  const uint32_t idesc = umma_idesc(128, 128, false);
  for (int kb = 0; kb < kScKBlocks; ++kb) {
    const int st = kb % kScStages;
    cp_async_wait<1>();
    fence_proxy_async_smem();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t sa = smem_u32(base + st * kScStage), sb = sa + 16384;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tmem, umma_desc(sa + ks * 32, 16, 1024, 2), umma_desc(sb + ks * 32, 16, 1024, 2), idesc,
                  (kb | ks) != 0);
      umma_commit(smem_u32(&bars[st]));
    }
    if (kb + 2 < kScKBlocks) {
      const int nst = (kb + 2) % kScStages;
      if (kb >= 1) mbar_wait(smem_u32(&bars[nst]), ((kb - 1) / kScStages) & 1, a.ws);  // MMAs of kb-1 done
      fill(kb + 2, nst);
    }
    cp_async_commit();
  }
  mbar_wait(smem_u32(&bars[(kScKBlocks - 1) % kScStages]), ((kScKBlocks - 1) / kScStages) & 1, a.ws);
  tc_fence_after();
  float mx = -INFINITY;
#pragma unroll
  for (int c0 = 0; c0 < 128; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(v[j]));
  }
  const int p = p0 + tid;  // this thread's tensor-memory lane = page row
  if (p < P) {
    const float sc = mx * a.scale;
    const bool forced = always_kept(p, P, a.sink, a.window);
    a.keys[(size_t)i * a.key_stride + p] = (row_blk[tid] >= 0 && !forced) ? score_key(sc) : 0u;
    if (a.scores_out) a.scores_out[(size_t)i * a.max_pages + p] = sc;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------------------------
// decode
// ------------------------------------------------------------------------------------
constexpr int kHalf = 32;                       // tokens per TMA box (half a tile)
constexpr int kTile = 64;                       // tokens per tile
constexpr int kQTmemKB = 6;                     // K blocks of Q held in tensor memory (dims 0..383)
constexpr int kQSmemKB = kKB - kQTmemKB;        // K blocks of Q in shared memory (dims 384..575)
constexpr int kQSBytes = kQSmemKB * kHeads * 128;  // 49152: 3 swizzled [128 x 64] blocks
constexpr int kKBlock = kTile * 128;            // 8192: one 64-dim block of a tile, 128-byte swizzle
constexpr int kKTile = kKB * kKBlock;           // 73728: a K tile (64 tokens x 576)
constexpr int kKStages = 2;
constexpr int kPBytes = kHeads * kTile * 2;     // 16384: P [128 x 64] bf16, 128-byte swizzle
constexpr int kDecSmem = 1024 + kQSBytes + kKStages * kKTile + kPBytes;
constexpr int kDecThreads = 192;                // 4 softmax warps (one thread per head), MMA warp, TMA warp
constexpr int kMlaMaxSw = 128;                  // pages per split
constexpr int kMlaMaxItems = 128;               // splits per (sequence, half); their merge weights fit the K stages
static_assert(kMlaMaxItems * kHeads * 4 <= kKStages * kKTile, "merge weights must fit the K stages");
// tensor-memory columns: O (128 x 256 fp32), S (128 x 64 fp32), Q dims 0..383 as bf16 pairs
constexpr uint32_t kOCol = 0, kSCol = 256, kQCol = 320;
static_assert(kQCol + kQTmemKB * 32 == 512, "tensor-memory budget");
constexpr float kRescaleSlack = 8.f;            // log2 headroom before O is rescaled
constexpr int kMlaClusterMax = 8;               // splits per (sequence, half) merged inside one cluster
constexpr int kORow = 256 + 4;                  // floats per parked O row (+4: conflict-free float4 reads)
static_assert(kHeads * kORow * 4 + kHeads * 8 + (kMlaClusterMax + 1) * kHeads * 4 <= kKStages * kKTile,
              "parked O rows, (m, l) and the merge weights must fit the K stages");

// One CTA per (split, half of D_v, sequence); warps 0-3 own one query head per thread (the
// tensor-memory lanes), warp 4's lane 0 issues every TMA copy and every MMA. A tcgen05.mma
// costs about the same to issue whatever its N up to 256, so S uses 64-token tiles (N = 64):
//   K(t)  : TMA (two 32-row boxes per 64-dim block) into stage t % 2   (kfull; freed after P.V(t))
//   S(t)  = Q K(t)^T (A = Q from tensor memory for dims 0..383, from shared memory for the rest)
//   P(t)  : softmax warps read S(t), rescale O when needed, write P(t)   (pready)
//   O    += P(t) V(t)   (V = the first 512 dims of K(t), MN-major)        (pvdone)
// in the order P.V(t), S(t+1), then the copy of K(t+2) into the stage P.V(t) released.
__global__ void __launch_bounds__(kDecThreads, 1) mla_decode_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmK) {
  pdl_wait();  // dependents are released when this grid completes
  extern __shared__ unsigned char dyn[];
  unsigned char *base = align1024(dyn);
  unsigned char *sQ = base;                    // Q dims 384..575
  unsigned char *sK = base + kQSBytes;         // kKStages K tiles
  unsigned char *sP = sK + kKStages * kKTile;  // P
  // K tile parts: A = the 64-dim blocks only S reads (free once S(t) is done), B = the four
  // value blocks of this half of D_v (free once P.V(t) is done)
  __shared__ __align__(8) uint64_t qbar, kfa[kKStages], kfb[kKStages], kea[kKStages], keb[kKStages], sfull, sfree,
      pready, pvdone, drained;
  __shared__ int abort_sh;  // set by the first wait that gives up: every later wait returns at once
  __shared__ uint32_t tslot;
  __shared__ int ent_blk[kMlaMaxSw], ent_valid[kMlaMaxSw];
  __shared__ short halves[2 * kMlaMaxSw];  // (entry, 32-token half) pairs with at least one live row
  __shared__ int n_halves_sh;
  __shared__ int flag_last;

  const int s = blockIdx.x, vh = blockIdx.y, i = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = i * 2 + vh;
  const size_t pbase = (size_t)unit * a.n_items_max + s;
  const int seq_len = a.seq_lens[i];
  const int P = (seq_len + a.ps - 1) / a.ps;
  const int e0 = s * a.sw;
  // the list loads do not depend on the length, so they go out with it (one list entry per
  // thread: sw <= kMlaMaxSw <= kDecThreads)
  const int32_t *row = a.selected ? a.selected + (size_t)i * a.b_max : nullptr;
  int first = -1, pg_x = e0 + tid, prev_x = -1;
  if (row && e0 < a.b_max) {
    first = row[e0];
    if (tid < a.sw && e0 + tid < a.b_max) {
      pg_x = row[e0 + tid];
      prev_x = e0 + tid > 0 ? row[e0 + tid - 1] : -1;
    }
  }
  // the block id of this thread's entry, requested as soon as its page id is known (in bounds of
  // the block table whatever the length; used only if the entry turns out valid), ahead of the
  // query loads below so that it does not queue behind them
  int blk_x = -1;
  if (tid < a.sw && pg_x >= 0 && pg_x < a.max_pages) blk_x = a.block_table[(size_t)i * a.max_pages + pg_x];
  // Q dims 0..383 of head `tid` go to tensor memory after the allocation below; its loads are
  // issued right behind the list and block-table loads above (volatile with a memory clobber, so
  // nothing moves across them), and land while the set-up runs (warps 0-3)
  constexpr int kQLd = kQTmemKB * 8;  // 16-byte loads in those dims
  const uint4 *qrow =
      reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(a.q) + ((size_t)i * kHeads + (tid & 127)) * kD);
  uint4 qv[kQLd];
  if (warp < 4) {
#pragma unroll
    for (int j = 0; j < kQLd; ++j)
      asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                   : "=r"(qv[j].x), "=r"(qv[j].y), "=r"(qv[j].z), "=r"(qv[j].w)
                   : "l"(qrow + j)
                   : "memory");
  }
  int n_ent = 0;
  if (seq_len < 1 || P > a.max_pages) {
    if (s == 0 && vh == 0 && tid == 0) set_status(a.ws, PSK_DEV_BAD_SEQLEN);
  } else if (row) {
    if (e0 < a.b_max && first >= 0) n_ent = min(a.sw, a.b_max - e0);
  } else if (e0 < P) {
    n_ent = min(a.sw, P - e0);
  }
  if (tid < n_ent) {
    int blk = -1;
    bool ok = true;
    if (row) {
      if (pg_x >= 0 && (pg_x >= P || pg_x <= prev_x || (e0 + tid > 0 && prev_x < 0))) {
        if (vh == 0) set_status(a.ws, PSK_DEV_BAD_SELECTED);
        ok = false;
      }
      if (pg_x < 0) ok = false;
    }
    if (ok) {
      blk = blk_x;
      if (blk < 0 || blk >= a.nb) {
        if (vh == 0) set_status(a.ws, PSK_DEV_BAD_BLOCK);
        ok = false;
      }
    }
    ent_blk[tid] = blk;
    ent_valid[tid] = ok ? min(a.ps, seq_len - pg_x * a.ps) : 0;
  }
  if (tid == 0) {
    mbar_init(smem_u32(&qbar), 1);
    mbar_init(smem_u32(&drained), 1);
    mbar_init(smem_u32(&sfull), 1);
    mbar_init(smem_u32(&sfree), 4);
    mbar_init(smem_u32(&pready), 4);
    mbar_init(smem_u32(&pvdone), 1);
    for (int k = 0; k < kKStages; ++k) {
      mbar_init(smem_u32(&kfa[k]), 1);
      mbar_init(smem_u32(&kfb[k]), 1);
      mbar_init(smem_u32(&kea[k]), 1);
      mbar_init(smem_u32(&keb[k]), 1);
    }
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  auto wait_ok = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (*reinterpret_cast<volatile int *>(&abort_sh)) return false;
    if (mbar_wait(smem_u32(bar), parity, a.ws)) return true;
    *reinterpret_cast<volatile int *>(&abort_sh) = 1;
    return false;
  };
  // the k-th 64-dim block S reads: part A (blocks outside this CTA's value half) first, then
  // part B (the value blocks vh * 4 .. vh * 4 + 3)
  auto s_block = [&](int k) -> int {
    const int kb = k < kKB - 4 ? k : (k - (kKB - 4)) + vh * 4;  // k >= 5: part B
    return k < kKB - 4 ? (kb < vh * 4 ? kb : kb + 4) : kb;
  };
  // Loading warp, before the others finish setting up: the (entry, 32-token half) pairs with at
  // least one live row in list order (a warp scan of each entry's 0-2 halves), then the copies
  // that wait for nothing (Q dims 384..575 and the first kKStages K tiles).
  int n_halves_l = 0, na = 0, nb = 0;  // loading warp: halves; part A / part B copies issued
  auto load_part = [&](int t, bool part_b) {
    const int st = t % kKStages;
    const int nh = (2 * t + 1 < n_halves_l) ? 2 : 1;
    const uint32_t bar = smem_u32(part_b ? &kfb[st] : &kfa[st]);
    const int nblk = part_b ? 4 : kKB - 4;
    mbar_arrive_expect_tx(bar, (uint32_t)(nh * nblk * kHalf * 128));
    const uint32_t dst = smem_u32(sK + st * kKTile);
    for (int h2 = 0; h2 < nh; ++h2) {
      const int hx = 2 * t + h2;
      const int e = halves[hx] >> 1, hh = halves[hx] & 1;
      const int row0 = ent_blk[e] * a.ps + hh * kHalf;
#pragma unroll 1
      for (int k = part_b ? kKB - 4 : 0; k < (part_b ? kKB : kKB - 4); ++k) {
        const int kb = s_block(k);
        tma_load_2d(dst + kb * kKBlock + h2 * kHalf * 128, &tmK, kb * 64, row0, bar);
      }
    }
  };
  if (warp == 5) {
    for (int eb = 0; eb < n_ent; eb += 32) {
      const int e = eb + lane;
      const int c = e < n_ent ? (ent_valid[e] + kHalf - 1) / kHalf : 0;  // halves with live rows
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      for (int hh = 0; hh < c; ++hh) halves[n_halves_l + incl - c + hh] = (short)(e * 2 + hh);
      n_halves_l += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    if (lane == 0) {
      n_halves_sh = n_halves_l;
      if (n_halves_l > 0) {
        mbar_arrive_expect_tx(smem_u32(&qbar), kQSBytes);
#pragma unroll 1
        for (int kb = 0; kb < kQSmemKB; ++kb)
          tma_load_2d(smem_u32(sQ + kb * kHeads * 128), &tmQ, (kQTmemKB + kb) * 64, i * kHeads, smem_u32(&qbar));
        const int t0 = min((n_halves_l + 1) / 2, kKStages);
        for (int t = 0; t < t0; ++t) {
          load_part(t, false);
          load_part(t, true);
        }
        na = nb = t0;
      }
    }
  }
  if (warp < 4 && n_ent > 0) {  // Q dims 0..383 of head `tid` into tensor memory (bf16 pairs)
#pragma unroll
    for (int c = 0; c < kQTmemKB; ++c) {
      uint32_t w[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        w[4 * j] = qv[c * 8 + j].x;
        w[4 * j + 1] = qv[c * 8 + j].y;
        w[4 * j + 2] = qv[c * 8 + j].z;
        w[4 * j + 3] = qv[c * 8 + j].w;
      }
      tmem_st32_async(tmem + lane_base + kQCol + c * 32, w);  // the six stores in flight together
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int n_halves = n_halves_sh;
  const int n_tiles = (n_halves + 1) / 2;
  // live rows of the two halves of tile t (0 for a missing second half)
  auto half_rows = [&](int hx) -> int {
    if (hx >= n_halves) return 0;
    const int e = halves[hx] >> 1, hh = halves[hx] & 1;
    return min(kHalf, ent_valid[e] - hh * kHalf);
  };
  float m_fin = -INFINITY, l_fin = 0.f;  // softmax warps: this head's (m, l) after the last tile
  if (warp == 5) {
    // ---------------- loading thread: TMA copies ----------------
    if (lane == 0 && n_tiles > 0) {  // tiles 0 .. kKStages - 1 went out before the set-up barrier
#pragma unroll 1
      for (int t = na; t < n_tiles; ++t) {
        const int st = t % kKStages;
        if (t >= kKStages && !wait_ok(&kea[st], ((t - kKStages) / kKStages) & 1)) break;  // S(t-2) done
        load_part(t, false);
        na = t + 1;
        if (t >= kKStages && !wait_ok(&keb[st], ((t - kKStages) / kKStages) & 1)) break;  // P.V(t-2) done
        load_part(t, true);
        nb = t + 1;
      }
      // every copy in flight lands before shared memory is released (also after a wait gave up)
      for (int t = max(0, na - kKStages); t < na; ++t) mbar_wait(smem_u32(&kfa[t % kKStages]), (t / kKStages) & 1, a.ws);
      for (int t = max(0, nb - kKStages); t < nb; ++t) mbar_wait(smem_u32(&kfb[t % kKStages]), (t / kKStages) & 1, a.ws);
      mbar_wait(smem_u32(&qbar), 0, a.ws);
    }
  } else if (warp == 4) {
    // ---------------- issuing thread: MMAs ----------------
    if (lane == 0 && n_tiles > 0) {
      bool ok = wait_ok(&qbar, 0);
      const uint32_t idesc_qk = umma_idesc(128, kTile, false);
      const uint32_t idesc_pv = umma_idesc(128, 256, true);
      // S(u) = Q K(u)^T in two parts: the blocks outside this CTA's value half (part A), then the
      // value blocks (part B); P.V of the previous tile is issued between them so that the value
      // blocks it frees can be refilled early. Descriptors advance by (bytes >> 4).
      const uint32_t q0 = smem_u32(sQ);
      auto issue_s_part = [&](int u, bool part_b) -> bool {
        const int st = u % kKStages;
        if (!wait_ok(part_b ? &kfb[st] : &kfa[st], (u / kKStages) & 1)) return false;
        tc_fence_after();
        const uint32_t d = tmem + kSCol;
        const uint32_t k0 = smem_u32(sK + st * kKTile);
#pragma unroll 1
        for (int k = part_b ? kKB - 4 : 0; k < (part_b ? kKB : kKB - 4); ++k) {
          const int kb = s_block(k);
          const uint64_t b0 = umma_desc(k0 + kb * kKBlock, 16, 1024, 2);
          if (kb < kQTmemKB) {
            const uint32_t a0 = tmem + kQCol + kb * 32;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16_ts(d, a0 + ks * 8, b0 + 2 * ks, idesc_qk, (k | ks) != 0);
          } else {
            const uint64_t a0 = umma_desc(q0 + (kb - kQTmemKB) * kHeads * 128, 16, 1024, 2);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16(d, a0 + 2 * ks, b0 + 2 * ks, idesc_qk, (k | ks) != 0);
          }
        }
        umma_commit(smem_u32(part_b ? &sfull : &kea[st]));
        return true;
      };
      auto issue_pv = [&](int t) -> bool {
        if (!wait_ok(&pready, t & 1)) return false;  // P(t) written, O rescaled
        tc_fence_after();
        const uint64_t pa = umma_desc(smem_u32(sP), 16, 1024, 2);
        const uint64_t vb = umma_desc(smem_u32(sK + (t % kKStages) * kKTile + vh * 4 * kKBlock), kKBlock, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // P: +32 bytes per 16 tokens; V: +16 rows of 128 bytes
          umma_bf16(tmem + kOCol, pa + 2 * ks, vb + 128 * ks, idesc_pv, (t | ks) != 0);
        umma_commit(smem_u32(&pvdone));
        umma_commit(smem_u32(&keb[t % kKStages]));
        return true;
      };
      ok = ok && issue_s_part(0, false) && issue_s_part(0, true);
#pragma unroll 1
      for (int t = 0; ok && t < n_tiles; ++t) {
        // all of S(t+1) as soon as the softmax warps hold S(t) in registers, so the tensor pipe
        // computes it while they turn S(t) into P(t); then P.V(t)
        if (t + 1 < n_tiles &&
            (!wait_ok(&sfree, t & 1) || !issue_s_part(t + 1, false) || !issue_s_part(t + 1, true)))
          break;
        if (!issue_pv(t)) break;
      }
      // every MMA issued completes before tensor memory and shared memory are released
      umma_commit(smem_u32(&drained));
      mbar_wait(smem_u32(&drained), 0, a.ws);
    }
  } else if (n_tiles > 0) {
    // ---------------- softmax warps: one query head per thread ----------------
    float m_run = -INFINITY, l_run = 0.f;
    const float qs = a.scale * kLog2e;
#pragma unroll 1
    for (int t = 0; t < n_tiles; ++t) {
      if (!__all_sync(0xffffffffu, wait_ok(&sfull, t & 1))) break;  // warp-uniform exit
      tc_fence_after();
      const int nva = half_rows(2 * t), nvb = half_rows(2 * t + 1);
      float x[kTile];
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + kSCol + c * 32, sv);
        const int nv = c == 0 ? nva : nvb;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[c * 32 + j] = j < nv ? __uint_as_float(sv[j]) * qs : -INFINITY;
          mt = fmaxf(mt, x[c * 32 + j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sfree));  // the issuing thread may overwrite S now
      // O holds P.V(t-1) and P is free once pvdone completes for t-1
      if (t > 0 && !__all_sync(0xffffffffu, wait_ok(&pvdone, (t - 1) & 1))) break;
      tc_fence_after();
      // The exponent reference m_run moves only when this head's max exceeds it by more than
      // kRescaleSlack (log2 units): p stays <= 2^kRescaleSlack, exact to fp32 rounding, and the
      // normaliser l uses the same reference, so the result is unchanged while the rescale of
      // O in tensor memory becomes rare. Tensor-memory loads and stores are warp-collective, so
      // a warp rescales together (alpha = 1 on lanes that keep their reference).
      const bool moved = t == 0 || mt > m_run + kRescaleSlack;
      const float m_new = moved ? fmaxf(m_run, mt) : m_run;
      const bool rescale = t > 0 && moved;
      if (__any_sync(0xffffffffu, rescale)) {
        const float al = rescale ? exp2f(m_run - m_new) : 1.f;
        l_run *= al;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kOCol + c0, ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * al);
          tmem_st32(tmem + lane_base + kOCol + c0, ov);
        }
      }
      m_run = m_new;
      // P row r = tid: 8 chunks of 16 bytes, 128-byte swizzle
      unsigned char *prow = sP + tid * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t pw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p0 = exp2f(x[c * 8 + 2 * j] - m_run), p1 = exp2f(x[c * 8 + 2 * j + 1] - m_run);
          l_run += p0 + p1;
          pw[j] = (uint32_t)f32_to_bf16_bits(p0) | ((uint32_t)f32_to_bf16_bits(p1) << 16);
        }
        *reinterpret_cast<uint4 *>(prow + ((c ^ (tid & 7)) * 16)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      }
      // Rows past the live tokens (the tail page past seq_len, or a missing second half) hold
      // whatever the stage last received; their P is 0, but 0 * NaN is NaN, so the value rows
      // this CTA multiplies are zeroed (128 bytes per row and 64-dim block).
      if (nva < kHalf || nvb < kHalf) {
        unsigned char *vblk = sK + (t % kKStages) * kKTile + vh * 4 * kKBlock;
        for (int x2 = tid; x2 < 4 * kTile * 8; x2 += kHeads) {
          const int kb = x2 / (kTile * 8), r = (x2 / 8) % kTile, c = x2 % 8;
          const bool live = r < kHalf ? r < nva : (r - kHalf) < nvb;
          if (!live) *reinterpret_cast<uint4 *>(vblk + kb * kKBlock + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&pready));
    }
    __all_sync(0xffffffffu, wait_ok(&pvdone, (n_tiles - 1) & 1));
    m_fin = m_run;
    l_fin = l_run;
  }

  // ---- the splits of a (sequence, half) merge ------------------------------------------------
  // Launched as one cluster per (sequence, half) (at most kMlaClusterMax splits), each CTA parks
  // its unnormalised O rows and (m, l) in its own shared memory (the K stages are free now) and
  // merges one slice of the value dims over distributed shared memory. Otherwise the partials
  // go to the workspace and the last CTA to finish merges them.
  const uint32_t n_clu = cluster_size();
  const bool clustered = n_clu == (uint32_t)a.n_items_max;
  float *sO = reinterpret_cast<float *>(sK);                     // [128][kORow]
  float2 *sML = reinterpret_cast<float2 *>(sK + kHeads * kORow * 4);  // [128]
  __syncthreads();  // the loading and issuing threads' last waits are over: no copy or MMA in flight
  if (warp < 4) {
    tc_fence_after();
    if (clustered) {
      if (n_tiles > 0) {
        float *orow = sO + tid * kORow;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kOCol + c0, ov);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(orow + c0 + j) = make_float4(
                __uint_as_float(ov[j]), __uint_as_float(ov[j + 1]), __uint_as_float(ov[j + 2]), __uint_as_float(ov[j + 3]));
        }
      }
      sML[tid] = make_float2(m_fin, l_fin);
    } else {
      if (n_tiles > 0) {  // partial O row (unnormalised) of head `tid`
        float *po = a.part_o + (pbase * kHeads + tid) * 256;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kOCol + c0, ov);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(po + c0 + j) = make_float4(
                __uint_as_float(ov[j]), __uint_as_float(ov[j + 1]), __uint_as_float(ov[j + 2]), __uint_as_float(ov[j + 3]));
        }
      }
      a.part_ml[(pbase * kHeads + tid) * 2] = m_fin;
      a.part_ml[(pbase * kHeads + tid) * 2 + 1] = l_fin;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);

  if (clustered) {
    // one split per (sequence, half): a CTA barrier and this CTA's own addresses (no cluster launch)
    const bool multi = n_clu > 1;
    if (multi) cluster_sync_all();  // every CTA of the cluster has parked its rows
    else __syncthreads();
    const int n = (int)n_clu;
    const int r = (int)cluster_rank();
    const int span = ((256 + n - 1) / n + 3) & ~3;  // value dims this CTA writes (a multiple of 4)
    const int d0 = min(256, r * span), d1 = min(256, d0 + span);
    float *wts = reinterpret_cast<float *>(sK + kHeads * kORow * 4 + kHeads * 8);  // [kMlaClusterMax + 1][128]
    if (tid < kHeads) {  // the merge weights of head `tid` (and 1 / L in the last row)
      float mk[kMlaClusterMax], lk[kMlaClusterMax];
#pragma unroll
      for (int k = 0; k < kMlaClusterMax; ++k) {
        float2 ml = make_float2(-INFINITY, 0.f);
        if (k < n) ml = ld_dsmem_f2(multi ? dsmem_addr(smem_u32(&sML[tid]), (uint32_t)k) : smem_u32(&sML[tid]));
        mk[k] = ml.x;
        lk[k] = ml.y;
      }
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kMlaClusterMax; ++k) M = fmaxf(M, mk[k]);
      float L = 0.f;
#pragma unroll
      for (int k = 0; k < kMlaClusterMax; ++k) {
        const float w = mk[k] == -INFINITY ? 0.f : exp2f(mk[k] - M);  // 0 for every k >= n
        if (w > 0.f) L = fmaf(w, lk[k], L);
        wts[k * kHeads + tid] = w;
      }
      wts[kMlaClusterMax * kHeads + tid] = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    if (warp < 4) {
      // each half-warp takes one head row and 16 consecutive float4 of it, so a warp's remote
      // loads are two contiguous 256-byte runs; four head pairs per step keep 4n loads in flight
      const int hl = lane >> 4, l16 = lane & 15;
      uint16_t *out_i = reinterpret_cast<uint16_t *>(a.out) + (size_t)i * kHeads * kDv + vh * 256;
#pragma unroll 1
      for (int pb = warp; pb < kHeads / 2; pb += 16) {
#pragma unroll 1
        for (int d = d0 + l16 * 4; d < d1; d += 64) {
          float4 o[4][kMlaClusterMax];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int h = 2 * (pb + 4 * u) + hl;
            const uint32_t src = smem_u32(sO + h * kORow + d);
#pragma unroll
            for (int k = 0; k < kMlaClusterMax; ++k)
              o[u][k] = wts[k * kHeads + h] != 0.f ? ld_dsmem_f4(multi ? dsmem_addr(src, (uint32_t)k) : src)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int h = 2 * (pb + 4 * u) + hl;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kMlaClusterMax; ++k) {
              const float w = wts[k * kHeads + h];
              if (w == 0.f) continue;
              acc.x = fmaf(w, o[u][k].x, acc.x);
              acc.y = fmaf(w, o[u][k].y, acc.y);
              acc.z = fmaf(w, o[u][k].z, acc.z);
              acc.w = fmaf(w, o[u][k].w, acc.w);
            }
            const float inv = wts[kMlaClusterMax * kHeads + h];
            uint2 wv;
            wv.x = (uint32_t)f32_to_bf16_bits(acc.x * inv) | ((uint32_t)f32_to_bf16_bits(acc.y * inv) << 16);
            wv.y = (uint32_t)f32_to_bf16_bits(acc.z * inv) | ((uint32_t)f32_to_bf16_bits(acc.w * inv) << 16);
            *reinterpret_cast<uint2 *>(out_i + (size_t)h * kDv + d) = wv;
          }
        }
      }
    }
    if (multi) cluster_sync_all();  // no CTA leaves while another still reads its shared memory
    return;
  }

  __threadfence();
  __syncthreads();
  if (tid == 0) flag_last = atomicAdd(a.tickets + unit, 1u) == (unsigned)(a.n_items_max - 1);
  __syncthreads();
  if (!flag_last || tid >= kHeads) return;
  __threadfence();
  if (tid == 0) a.tickets[unit] = 0u;
  const size_t it0 = (size_t)unit * a.n_items_max;
  float *wsm = reinterpret_cast<float *>(sK);  // [n_items][128] merge weights (stages are free now)
  float M = -INFINITY;
  for (int k = 0; k < a.n_items_max; ++k) M = fmaxf(M, __ldcg(a.part_ml + ((it0 + k) * kHeads + tid) * 2));
  float L = 0.f;
  for (int k = 0; k < a.n_items_max; ++k) {
    const float mk = __ldcg(a.part_ml + ((it0 + k) * kHeads + tid) * 2);
    const float w = mk == -INFINITY ? 0.f : exp2f(mk - M);
    if (w > 0.f) L = fmaf(w, __ldcg(a.part_ml + ((it0 + k) * kHeads + tid) * 2 + 1), L);
    wsm[k * kHeads + tid] = w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint16_t *out = reinterpret_cast<uint16_t *>(a.out) + ((size_t)i * kHeads + tid) * kDv + vh * 256;
  // four splits' 32-dim slices in flight at once (a walk over the splits one at a time waited a
  // full L2 round trip per slice)
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
#pragma unroll 1
    for (int k0 = 0; k0 < a.n_items_max; k0 += 4) {
      float4 o[4][8];
      float w4[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = k0 + kk;
        w4[kk] = k < a.n_items_max ? wsm[k * kHeads + tid] : 0.f;
        const float4 *pk = reinterpret_cast<const float4 *>(a.part_o + ((it0 + k) * kHeads + tid) * 256 + c * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[kk][j] = w4[kk] != 0.f ? __ldcg(pk + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (w4[kk] == 0.f) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[4 * j] = fmaf(w4[kk], o[kk][j].x, acc[4 * j]);
          acc[4 * j + 1] = fmaf(w4[kk], o[kk][j].y, acc[4 * j + 1]);
          acc[4 * j + 2] = fmaf(w4[kk], o[kk][j].z, acc[4 * j + 2]);
          acc[4 * j + 3] = fmaf(w4[kk], o[kk][j].w, acc[4 * j + 3]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      uint4 w;
      w.x = (uint32_t)f32_to_bf16_bits(acc[j] * inv) | ((uint32_t)f32_to_bf16_bits(acc[j + 1] * inv) << 16);
      w.y = (uint32_t)f32_to_bf16_bits(acc[j + 2] * inv) | ((uint32_t)f32_to_bf16_bits(acc[j + 3] * inv) << 16);
      w.z = (uint32_t)f32_to_bf16_bits(acc[j + 4] * inv) | ((uint32_t)f32_to_bf16_bits(acc[j + 5] * inv) << 16);
      w.w = (uint32_t)f32_to_bf16_bits(acc[j + 6] * inv) | ((uint32_t)f32_to_bf16_bits(acc[j + 7] * inv) << 16);
      *reinterpret_cast<uint4 *>(out + c * 32 + j) = w;
    }
  }
}

}  // namespace

bool mla_supported(const psk_layout &L) {
  return L.latent == 1 && L.dtype == PSK_BF16 && L.num_kv_heads == 1 && L.num_q_heads == kHeads && L.head_dim == kD &&
         L.v_head_dim == kDv && (L.page_size == 32 || L.page_size == 64);
}

size_t mla_qsplit_bytes(const psk_layout &L) { return (size_t)L.batch * kHeads * 2 * kD * 2; }

cudaError_t launch_mla_score_select(const ScoreArgs &a, uint16_t *qsplit, cudaStream_t s, int stages) {
  if (!(stages & kStageScore)) return launch_page_select(a, s, true);
  const int rows = a.B * kHeads;
  const int n = rows * (kD / 8);
  cudaError_t e = launch_kernel(true, mla_qsplit_kernel, (n + 255) / 256, 256, 0, s,
                                reinterpret_cast<const uint16_t *>(a.q), qsplit, rows);
  if (e != cudaSuccess) return e;
  dim3 grid((a.max_pages + 127) / 128, a.B);
  e = launch_kernel(false, mla_score_kernel, grid, 128, kScSmem, s, a, (const uint16_t *)qsplit);
  if (e != cudaSuccess || !(stages & kStageSelect)) return e;
  return launch_page_select(a, s);
}

bool plan_mla_decode(const psk_layout &L, int entries, DecodePlan *plan) {
  const long long units = (long long)L.batch * 2;
  const long long sms = sm_count();
  // One CTA per SM (shared memory). Pick the split width that minimises
  //   waves * (pages per split + ~2 pages of fixed per-CTA cost) + the merge,
  // where a merge inside one cluster (at most kMlaClusterMax splits) costs about a page and the
  // workspace merge about a page per split (measured on the latent workload: 4 splits merged by
  // the last CTA took 52 us before its loads were batched, about 20 pages).
  int sw = std::max(1, std::min(entries, kMlaMaxSw));
  double best = 1e300;
  for (int items = 1; items <= std::min(std::max(entries, 1), kMlaMaxItems); ++items) {
    const int w = (std::max(entries, 1) + items - 1) / items;
    if (w > kMlaMaxSw) continue;
    const int n = (std::max(entries, 1) + w - 1) / w;
    const long long waves = (units * n + sms - 1) / sms;
    const double cost = (double)waves * (w + 2.0) + (n <= kMlaClusterMax ? 1.0 : 1.0 * n);
    if (cost < best - 1e-9) {
      best = cost;
      sw = w;
    }
  }
  plan->sw = sw;
  plan->n_items_max = (entries + sw - 1) / sw;
  size_t off = ws_scratch_offset((size_t)units);
  plan->off_o = off;
  off = align_up(off + (size_t)units * plan->n_items_max * kHeads * 256 * 4, 256);
  plan->off_ml = off;
  off = align_up(off + (size_t)units * plan->n_items_max * kHeads * 2 * 4, 256);
  plan->ws_bytes = off;
  plan->off_tickets = ws_decode_tickets_offset((size_t)units);
  plan->flat = 0;
  plan->taper = 0;
  plan->off_counts = 0;
  return plan->n_items_max <= kMlaMaxItems;
}

// PSK_MLA_CLUSTER=0: the latent decode without clusters (its splits then merge in the workspace,
// with the same arithmetic in the same order); read once per process
bool mla_cluster_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("PSK_MLA_CLUSTER");
    return !(v && v[0] == '0');
  }();
  return on;
}

cudaError_t launch_mla_decode(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap tmQ, tmK;
  if (!encode_matrix_map_sw128(&tmQ, a.q, kD, (long long)a.B * kHeads, 64, kHeads) ||
      !encode_matrix_map_sw128(&tmK, a.k_cache, kD, (long long)a.nb * a.ps, 64, kHalf))
    return cudaErrorInvalidValue;
  dim3 grid(a.n_items_max, 2, a.B);
  if (a.n_items_max > 1 && a.n_items_max <= kMlaClusterMax && mla_cluster_enabled()) {
    // the splits of each (sequence, half) as one cluster: they merge in distributed shared memory
    const void *fn = reinterpret_cast<const void *>(mla_decode_kernel);
    cudaError_t e = kernel_setup(fn, kDecThreads, kDecSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = kDecSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.n_items_max;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled(true) ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, mla_decode_kernel, a, tmQ, tmK) == cudaSuccess) return cudaSuccess;
    (void)cudaGetLastError();  // clusters of this size cannot be placed: the workspace merge below
  }
  return launch_kernel(true, mla_decode_kernel, grid, kDecThreads, kDecSmem, s, a, tmQ, tmK);
}

}  // namespace psk
