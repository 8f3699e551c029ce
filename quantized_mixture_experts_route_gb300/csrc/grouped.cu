// grouped.cu -- grouped per-expert dequant-GEMM path (tcgen05, sm_103a).
#include "qmoe_internal.cuh"

namespace qmoe {

cudaError_t launch_grouped(const Problem&, bool, const uint8_t*, const void*, const uint8_t*,
                           const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace qmoe
