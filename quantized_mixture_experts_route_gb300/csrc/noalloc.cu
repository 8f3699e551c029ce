// qmoe_forward_decode_static: the decode-path layer forward with its workspace in
// a fixed device array of this library instead of a caller-provided buffer, for
// callers that cannot allocate device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds QMOE_STATIC_WORKSPACE_BYTES of it until the process exits. In
// host code its name is only a stand-in: the device address comes from
// cudaGetSymbolAddress, taken once per device (with that device current) at the
// first call on that device and cached. All calls on a device share the array
// and it keeps the previous call's contents, so the counters and the split-K
// tickets, which must start at zero, are cleared on the stream first. Calls
// whose work overlaps on the GPU (other streams, other threads) race on the array.
// Nothing here allocates device memory.
#include <mutex>

#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

constexpr int kMaxStaticDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[QMOE_STATIC_WORKSPACE_BYTES];

std::mutex g_static_mu;
void* g_static_ptr[kMaxStaticDevices] = {};

// Device address of g_static_workspace on the current device (set up on first use).
cudaError_t static_workspace(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (err != cudaSuccess) return err;
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
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
  const bool decode = p->path == QMOE_PATH_DECODE || (p->path == QMOE_PATH_AUTO && p->T <= kDecodeMaxT);
  if (!decode) return QMOE_ERR_UNSUPPORTED;
  if (need > QMOE_STATIC_WORKSPACE_BYTES) return QMOE_ERR_WORKSPACE_TOO_SMALL;

  void* base = nullptr;
  if (static_workspace(&base) != cudaSuccess) return QMOE_ERR_CUDA;
  Problem ip{};
  ip.T = p->T;
  ip.H = p->hidden;
  ip.I = p->inter;
  ip.E = p->num_experts;
  ip.k = p->top_k;
  ip.bits = p->bits;
  ip.block = p->block_size;
  ip.dtype = p->dtype;
  ip.path = QMOE_PATH_DECODE;
  Workspace ws;
  workspace_layout(ip, false, base, &ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws.counters, 0, sizeof(int32_t) * 4, s) != cudaSuccess) return QMOE_ERR_CUDA;
  if (ws.dunits_max > 0 &&
      cudaMemsetAsync(ws.dticket, 0, sizeof(int32_t) * ws.dunits_max, s) != cudaSuccess)
    return QMOE_ERR_CUDA;
  return qmoe_forward(p, x, router_logits, fc1_q, fc1_scales, fc1_zp, fc2_q, fc2_scales, fc2_zp, out,
                      base, QMOE_STATIC_WORKSPACE_BYTES, stream);
}
