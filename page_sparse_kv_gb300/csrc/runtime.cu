// Host-side launch facts, computed once and cached: whether launches carry the programmatic
// dependent-launch attribute, each device's SM count, each kernel's shared-memory limit and
// occupancy, and the tuning overrides from the environment. The C ABI's calls run these checks on
// every launch, so after the first call of a process they cost a table lookup instead of driver
// queries.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "psk_common.cuh"

namespace psk {

bool pdl_enabled(bool first_of_call) {
  static const int mode = [] {
    const char *env = std::getenv("PSK_PDL");
    return env ? std::atoi(env) : 1;
  }();
  return mode == 1 || (mode == 2 && !first_of_call);
}

namespace {
constexpr int kMaxDevices = 64;
constexpr int kDefaultSms = 152;  // used only by host-side size queries on a machine without a GPU

struct KernelEntry {
  int dev;
  const void *fn;
  size_t smem_set;       // dynamic shared-memory limit set on the kernel (0: not yet)
  int threads;           // occupancy cached for (threads, occ_smem)
  size_t occ_smem;
  int per_sm;            // -1: not yet computed
};

std::mutex g_mu;
std::vector<KernelEntry> g_kernels;
int g_sms[kMaxDevices] = {};

KernelEntry &entry(int dev, const void *fn) {
  for (auto &k : g_kernels)
    if (k.dev == dev && k.fn == fn) return k;
  g_kernels.push_back({dev, fn, 0, 0, 0, -1});
  return g_kernels.back();
}
}  // namespace

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return kDefaultSms;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      return kDefaultSms;
    }
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

cudaError_t kernel_setup(const void *fn, int threads, size_t smem, int *per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  KernelEntry &k = entry(dev, fn);
  // dynamic + static shared memory above 48 KB needs the opt-in: set it for any dynamic size
  if (smem > 0 && k.smem_set < smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k.smem_set = smem;
  }
  if (per_sm) {
    if (k.per_sm < 0 || k.threads != threads || k.occ_smem != smem) {
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
      if (e != cudaSuccess) return e;
      k.per_sm = n;
      k.threads = threads;
      k.occ_smem = smem;
    }
    *per_sm = k.per_sm;
  }
  return cudaSuccess;
}

void kernel_forget(const void *fn) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto &k : g_kernels)
    if (k.dev == dev && k.fn == fn) {
      k.smem_set = 0;
      k.per_sm = -1;
    }
}

const Tuning &tuning() {
  static const Tuning t = [] {
    Tuning r;
    if (const char *v = std::getenv("PSK_SCORE_TAIL")) r.score_tail = std::atoll(v);
    if (const char *v = std::getenv("PSK_SCORE_TAIL_CHUNK")) {
      const int x = std::atoi(v);
      if (x >= 1 && x <= 4096) r.score_tail_chunk = x;
    }
    if (const char *v = std::getenv("PSK_SCORE_PCHUNK")) {
      const int x = std::atoi(v);
      if (x >= 8 && x <= 4096) r.score_pchunk = x;
    }
    if (const char *v = std::getenv("PSK_SELECT_CHUNK")) {
      const int x = std::atoi(v);
      if (x >= 1024 && x <= 16384 && (x & (x - 1)) == 0) r.select_chunk = x;
    }
    if (const char *v = std::getenv("PSK_SCORE_MMA")) r.score_mma = std::atoi(v) != 0;
    if (const char *v = std::getenv("PSK_DECODE_MMA")) r.decode_mma = std::atoi(v) != 0;
    if (const char *v = std::getenv("PSK_DECODE_LAYOUT")) r.decode_layout = !std::strcmp(v, "split") ? 1 : (!std::strcmp(v, "flat") ? 2 : 0);
    if (const char *v = std::getenv("PSK_DECODE_SPLIT")) r.decode_split = std::atoi(v);
    r.decode_no_taper = std::getenv("PSK_DECODE_NO_TAPER") != nullptr;
    return r;
  }();
  return t;
}

}  // namespace psk
