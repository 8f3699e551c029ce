// combine.cu -- routing-weighted combine, one FP32 sum rounded once (sm_103a).
//
// out[t, :] = round(sum_{j<k} y_w[t*k + j, :]) where y_w already carries the
// routing weight (multiplied in the fc2 epilogue). The sum runs in FP32 in
// ascending j, is rounded to BF16/FP16 exactly once with round-to-nearest-even,
// and NaN stays NaN ("[CUDA] Add MoEPacked CPU/GPU hybrid offload ..." #33973:
// the partial sum stays in FP32 and is rounded once, as the GPU-only finalize
// does; "Keep NaN as NaN when rounding to BF16"). Routes whose weight is exactly
// zero are skipped ("skip zero-scale routes in the prefill finalizer", same PR).
// With an FC2 bias b2 [E][H] the sum adds w_j * b2[expert of route j] next to
// each route's row (the bias is applied per route, before the weight's sum and
// the one rounding: "[CUDA] Add INT4 and INT3 QMoE CPU/GPU offload support"
// #33575, commit notes).
// Memory bound: each thread reads k x 32 bytes and writes 16 bytes.
#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(Problem p, Workspace ws,
                                                      uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int per_row = p.H / 8;
  const int64_t total = p.T * per_row;
  // a matmul kernel of this call gave up on a wait: no plausible numbers
  const bool failed = *reinterpret_cast<volatile const int*>(ws.counters + 2) != 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_row;
    const int h0 = (int)(i % per_row) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // routes in batches of 8: every load of a batch is issued before the first add
    for (int j0 = 0; j0 < p.k; j0 += 8) {
      float w[8];
      float4 a[8], b[8];
      int ex[8];
      uint4 bbv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = j0 + j < p.k ? ws.topk_w[t * p.k + j0 + j] : 0.0f;
      if (p.b2)
#pragma unroll
        for (int j = 0; j < 8; ++j) ex[j] = ws.topk_idx[t * p.k + (j0 + j < p.k ? j0 + j : j0)];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t r = t * p.k + (j0 + j < p.k ? j0 + j : j0);
        const float4* src = reinterpret_cast<const float4*>(ws.y + r * p.H + h0);
        a[j] = src[0];
        b[j] = src[1];
      }
      // the batch's FC2 bias rows, all issued before the first is used (each waits
      // for its route's expert only)
      if (p.b2)
#pragma unroll
        for (int j = 0; j < 8; ++j) bbv[j] = *reinterpret_cast<const uint4*>(p.b2 + (int64_t)ex[j] * p.H + h0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (w[j] == 0.0f) continue;   // also the batch's padding past k
        if (p.b2) {
          const uint4 bb = bbv[j];
          const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
          float bv[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            bv[2 * q] = half_bits_to_float((uint16_t)(bw[q] & 0xFFFFu), p.dtype);
            bv[2 * q + 1] = half_bits_to_float((uint16_t)(bw[q] >> 16), p.dtype);
          }
          acc[0] += a[j].x + w[j] * bv[0]; acc[1] += a[j].y + w[j] * bv[1];
          acc[2] += a[j].z + w[j] * bv[2]; acc[3] += a[j].w + w[j] * bv[3];
          acc[4] += b[j].x + w[j] * bv[4]; acc[5] += b[j].y + w[j] * bv[5];
          acc[6] += b[j].z + w[j] * bv[6]; acc[7] += b[j].w + w[j] * bv[7];
          continue;
        }
        acc[0] += a[j].x; acc[1] += a[j].y; acc[2] += a[j].z; acc[3] += a[j].w;
        acc[4] += b[j].x; acc[5] += b[j].y; acc[6] += b[j].z; acc[7] += b[j].w;
      }
    }
    if (failed)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = __int_as_float(0x7FC00000);
    uint4 o;
    o.x = float_to_half_bits(acc[0], p.dtype) | ((uint32_t)float_to_half_bits(acc[1], p.dtype) << 16);
    o.y = float_to_half_bits(acc[2], p.dtype) | ((uint32_t)float_to_half_bits(acc[3], p.dtype) << 16);
    o.z = float_to_half_bits(acc[4], p.dtype) | ((uint32_t)float_to_half_bits(acc[5], p.dtype) << 16);
    o.w = float_to_half_bits(acc[6], p.dtype) | ((uint32_t)float_to_half_bits(acc[7], p.dtype) << 16);
    *reinterpret_cast<uint4*>(out + t * p.H + h0) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const Problem& p, const Workspace& ws, void* out, cudaStream_t s) {
  const int sms = device_sm_count();
  const int64_t total = p.T * (p.H / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  return launch_pdl(combine_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p, ws, static_cast<uint16_t*>(out));
}

}  // namespace qmoe
