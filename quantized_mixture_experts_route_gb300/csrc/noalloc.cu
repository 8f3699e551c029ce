// qmoe_forward_decode_static: the decode-path layer forward with its workspace in
// a fixed device array of this library instead of a caller-provided buffer, for
// callers that cannot allocate device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds QMOE_STATIC_WORKSPACE_BYTES of it until the process exits. In
// host code its name is only a stand-in: the device address comes from
// cudaGetSymbolAddress, taken on the first call made with a given device and
// context current, and cached for that pair (a context created after
// cudaDeviceReset gets its own look-up). All calls on a device share the array
// and it keeps the previous call's contents. What must start at zero -- the
// routing counters, the failure word, the split-K tickets and the decode layer
// kernel's claim and arrival counters -- is reset by the routing kernel at the
// start of every decode-path call, so nothing is cleared here. Calls whose work
// overlaps on the GPU (other streams, other threads) race on the array.
// Nothing here allocates device memory.
#include <map>
#include <mutex>
#include <utility>

#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[QMOE_STATIC_WORKSPACE_BYTES];

std::mutex g_static_mu;
std::map<std::pair<int, const void*>, void*> g_static_ptr;   // (device, context) -> address

// Device address of g_static_workspace on the current device and context (set
// up on first use there).
cudaError_t static_workspace(void** out) {
  int dev = 0;
  const void* ctx = nullptr;
  if (!current_device_context(&dev, &ctx)) return cudaErrorNoDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  auto it = g_static_ptr.find({dev, ctx});
  if (ctx && it != g_static_ptr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* ptr = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&ptr, g_static_workspace);
  if (err != cudaSuccess) return err;
  // the look-up makes the device's context current if none was: key the entry by it
  if (!ctx && !current_device_context(&dev, &ctx)) return cudaErrorNoDevice;
  g_static_ptr[{dev, ctx}] = ptr;
  *out = ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace qmoe

using namespace qmoe;

extern "C" qmoe_status qmoe_forward_decode_static(const qmoe_problem* p, const void* x,
                                                  const void* router_logits, const uint8_t* fc1_q,
                                                  const void* fc1_scales, const uint8_t* fc1_zp,
                                                  const uint8_t* fc2_q, const void* fc2_scales,
                                                  const uint8_t* fc2_zp, void* out, void* stream) {
  if (!p) return QMOE_ERR_INVALID_ARGUMENT;
  const size_t need = qmoe_workspace_bytes(p);
  // an invalid problem, or T == 0: qmoe_forward reports it without touching the GPU
  if (need == 0 || p->T == 0)
    return qmoe_forward(p, x, router_logits, fc1_q, fc1_scales, fc1_zp, fc2_q, fc2_scales, fc2_zp,
                        out, nullptr, 0, stream);
  const bool decode = resolve_path(*p) == QMOE_PATH_DECODE;
  if (!decode) return QMOE_ERR_UNSUPPORTED;
  if (need > QMOE_STATIC_WORKSPACE_BYTES) return QMOE_ERR_WORKSPACE_TOO_SMALL;

  void* base = nullptr;
  if (static_workspace(&base) != cudaSuccess) return QMOE_ERR_CUDA;
  return qmoe_forward(p, x, router_logits, fc1_q, fc1_scales, fc1_zp, fc2_q, fc2_scales, fc2_zp, out,
                      base, QMOE_STATIC_WORKSPACE_BYTES, stream);
}
