// launch_cache.cu -- per-device launch facts: SM count and the dynamic
// shared-memory opt-in of each kernel.
//
// Both belong to a device's context, not to the process: a process that drives
// several GPUs (one replica per device, from one or several host threads) needs
// the opt-in once on every device, and a context created after cudaDeviceReset
// starts without it. Entries are therefore keyed by (device ordinal, current
// context) and guarded by one mutex, so concurrent calls on different streams
// or devices are safe.
#include <cuda.h>

#include <map>
#include <mutex>
#include <tuple>

#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, resolved at run time (the library does not link
// the driver library).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

struct Key {
  int dev;
  const void* ctx;
  bool operator<(const Key& o) const { return std::tie(dev, ctx) < std::tie(o.dev, o.ctx); }
};

std::mutex g_mu;
std::map<Key, int> g_sms;
std::map<std::pair<Key, const void*>, int> g_smem;

// The calling thread's device and current context. Before the runtime has made
// a context current the context part is null; the entry made then is simply
// not found again once a context exists, and the fact is looked up once more.
bool current_key(Key* k) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  CUcontext ctx = nullptr;
  if (auto fn = ctx_get_current()) fn(&ctx);
  *k = Key{dev, ctx};
  return true;
}

}  // namespace

bool current_device_context(int* dev, const void** ctx) {
  Key k;
  if (!current_key(&k)) return false;
  *dev = k.dev;
  *ctx = k.ctx;
  return true;
}

int device_sm_count() {
  Key k;
  if (!current_key(&k)) return 148;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_sms.find(k);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, k.dev) != cudaSuccess || n <= 0) n = 148;
  g_sms[k] = n;
  return n;
}

cudaError_t ensure_smem_optin(const void* fn, int bytes) {
  Key k;
  if (!current_key(&k)) return cudaErrorNoDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  int& have = g_smem[{k, fn}];
  if (have >= bytes) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) have = bytes;
  return err;
}

}  // namespace qmoe
