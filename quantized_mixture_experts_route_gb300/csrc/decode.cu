// decode.cu -- decode path (T <= 8): split-K dequant-GEMV kernels (sm_103a).
//
// For each expert that received routes, the selected expert's packed weight
// rows are streamed from HBM once with wide vector loads (16/12/8 bytes of codes
// per lane per row), dequantised in registers and multiplied with the <= 8
// routed activation rows. The pages' decode kernels (MoeGemvTcInt4Kernel,
// FusedFc1FastVecKernel / Fc2RouteFastVecKernel, "[CUDA] Enable Tensor-Core
// INT3/INT4 QMoE offload ..." #33731) group <= 8 routes of one expert per CTA and
// use an m16n8k16 tensor-core step; this kernel keeps that grouping because the
// eight routes of a T <= 8 batch fit one MMA N-fragment, so every weight byte is
// read exactly once per call and the tensor core does the multiply-adds.
//
// Work split. A CTA owns 16 weight rows of one active expert and splits K over
// KSPLIT warps; the partial tiles are added in a fixed warp order (no atomics),
// so results are bit-reproducible. A quad of lanes covers 128 consecutive K of
// two rows (g, g+8) per chunk: lane c takes codes [32c, 32c+32) of the chunk.
//
// Numerics. A weight is (code - zp) * scale: with the code placed in the
// mantissa of FP16 1024.0, one exact FP16 subtraction gives (code - zp) and one
// FP16 multiplication by the scale is exact for BF16 scales in the FP16 normal
// range (at most 11 significant bits). Activations arrive as FP16 scaled by a
// power of two per token; the MMA accumulates in FP32.
//
// fc1 epilogue: h_i = silu(gate_i) * up_i from the interleaved rows 2i / 2i+1
// (activation_type "swiglu", swiglu_fusion = 1), stored in FP16 with the
// token's power of two squared. fc2 epilogue: y = (W2 h) / scale^2 * w_route in
// FP32, stored per route id for the combine.
#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

constexpr int kRowsPerCta = 16;
constexpr int kMaxKsplit = 8;
constexpr int kChunkK = 128;      // K covered by one quad of lanes per step
constexpr int kChunksPerBatch = 2;

template <int BITS>
struct Codes {
  uint32_t w[BITS];  // 32 codes of one row: 4 words (INT4), 3 (INT3), 2 (INT2)
};

template <int BITS>
__device__ __forceinline__ Codes<BITS> load_codes(const uint8_t* p) {
  Codes<BITS> c;
  if constexpr (BITS == 4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    c.w[0] = v.x; c.w[1] = v.y; c.w[2] = v.z; c.w[3] = v.w;
  } else if constexpr (BITS == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    c.w[0] = v.x; c.w[1] = v.y;
  } else {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
    c.w[0] = __ldg(q); c.w[1] = __ldg(q + 1); c.w[2] = __ldg(q + 2);
  }
  return c;
}

__device__ __forceinline__ uint32_t h2_sub_mul(uint32_t biased, uint32_t zp2, uint32_t s2) {
  const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&biased),
                                    *reinterpret_cast<const __half2*>(&zp2)),
                            *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The 16 FP16 pairs of a lane's 32 codes, in the K-order permutation of the
// activations (pair p holds stored positions 2p and 2p+1).
template <int BITS>
__device__ __forceinline__ void dequant_pairs(const Codes<BITS>& c, uint32_t zp2, uint32_t s2,
                                              uint32_t* pr) {
  constexpr uint32_t kMagic = 0x64006400u;  // FP16 1024.0 in both halves
  if constexpr (BITS == 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m)
        pr[4 * i + m] = h2_sub_mul(((c.w[i] >> (4 * m)) & 0x000F000Fu) | kMagic, zp2, s2);
  } else if constexpr (BITS == 2) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int m = 0; m < 8; ++m)
        pr[8 * i + m] = h2_sub_mul(((c.w[i] >> (2 * m)) & 0x00030003u) | kMagic, zp2, s2);
  } else {
    // groups of eight 3-bit codes: G0 = bytes 0-2, G1 = 3-5, G2 = 6-8, G3 = 9-11.
    // Pair (G0_m, G1_m) and (G2_m, G3_m) need the two groups' bits in the two
    // 16-bit halves: gather them with byte permutes.
    const uint32_t lo0 = __byte_perm(c.w[0], c.w[1], 0x4310);  // G0 bits 0-15 | G1 bits 0-15
    const uint32_t hi0 = __byte_perm(c.w[0], c.w[1], 0x5421);  // G0 bits 8-23 | G1 bits 8-23
    const uint32_t lo1 = __byte_perm(c.w[1], c.w[2], 0x6532);  // G2 bits 0-15 | G3 bits 0-15
    const uint32_t hi1 = __byte_perm(c.w[1], c.w[2], 0x7643);  // G2 bits 8-23 | G3 bits 8-23
#pragma unroll
    for (int m = 0; m < 5; ++m) {
      pr[m] = h2_sub_mul(((lo0 >> (3 * m)) & 0x00070007u) | kMagic, zp2, s2);
      pr[8 + m] = h2_sub_mul(((lo1 >> (3 * m)) & 0x00070007u) | kMagic, zp2, s2);
    }
#pragma unroll
    for (int m = 5; m < 8; ++m) {
      pr[m] = h2_sub_mul(((hi0 >> (3 * m - 8)) & 0x00070007u) | kMagic, zp2, s2);
      pr[8 + m] = h2_sub_mul(((hi1 >> (3 * m - 8)) & 0x00070007u) | kMagic, zp2, s2);
    }
  }
}

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t scale_half2(uint16_t bits, int dtype) {
  uint16_t h = bits;
  if (dtype == QMOE_BF16) h = __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)bits << 16)));
  return (uint32_t)h | ((uint32_t)h << 16);
}

__device__ __forceinline__ uint32_t zp_half2(const uint8_t* zp, int64_t idx, int bits) {
  const uint32_t z = zp ? (uint32_t)zp[idx] : (1u << (bits - 1));
  const uint32_t h = 0x6400u + z;  // FP16 1024 + z
  return h | (h << 16);
}

struct DecodeArgs {
  const uint8_t* q;        // [E][N][K*bits/8]
  const uint16_t* s;       // [E][N][K/block]
  const uint8_t* zp;       // [E][N][K/block] or null
  const uint16_t* act;     // FC1: x16 [T][K] by token; FC2: h16 [R][K] by sorted position
  int N, K;
  int ksplit;
  Problem p;
  Workspace ws;
};

// Index of h_j in the permuted FP16 row layout.
__device__ __forceinline__ int permuted_pos(int j, int G) {
  const int base = j - j % G, i = j % G;
  return base + (i < G / 2 ? 2 * i : 2 * (i - G / 2) + 1);
}

template <int BITS, bool FC1>
__global__ void __launch_bounds__(32 * kMaxKsplit) decode_gemv_kernel(DecodeArgs a) {
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  const int n_active = ws.counters[0];
  if ((int)blockIdx.y >= n_active) return;
  const int e = ws.active[blockIdx.y];
  const int begin = ws.offsets[e];
  const int n_e = ws.offsets[e + 1] - begin;  // <= 8 on this path
  const int K = a.K, N = a.N;
  const int nq = (K + kChunkK - 1) / kChunkK;
  const int row0 = blockIdx.x * kRowsPerCta;

  extern __shared__ __align__(16) uint8_t smem[];
  uint4* xs = reinterpret_cast<uint4*>(smem);  // [nq][4][32] x 16 bytes
  float* red = reinterpret_cast<float*>(smem + (size_t)nq * 4 * 32 * 16);  // [ksplit][32][4]
  float* tile = red + a.ksplit * 32 * 4;                                   // [16][8]

  // Activation rows of this expert's routes, in MMA B-fragment order.
  for (int P = threadIdx.x; P < nq * 128; P += blockDim.x) {
    const int q = P >> 7, i = (P >> 5) & 3, L = P & 31;
    const int n = L >> 2, c = L & 3;
    const int kk = q * kChunkK + 32 * c + 8 * i;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < n_e && kk < K) {
      const int pos = begin + n;
      const int64_t row = FC1 ? (int64_t)(ws.sorted_route[pos] / p.k) : (int64_t)pos;
      v = *reinterpret_cast<const uint4*>(a.act + row * K + kk);
    }
    xs[P] = v;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t rowA = (int64_t)e * N + row0 + g;
  const int64_t rowB = rowA + 8;
  const int64_t pitch = (int64_t)K * BITS / 8;
  const int nblk = K / p.block;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  for (int q0 = warp; warp < a.ksplit && q0 < nq; q0 += a.ksplit * kChunksPerBatch) {
    Codes<BITS> ca[kChunksPerBatch], cb[kChunksPerBatch];
    uint32_t sa[kChunksPerBatch], sb[kChunksPerBatch], za[kChunksPerBatch], zb[kChunksPerBatch];
    bool live[kChunksPerBatch];
#pragma unroll
    for (int u = 0; u < kChunksPerBatch; ++u) {
      const int q = q0 + u * a.ksplit;
      const int kk = q * kChunkK + 32 * c;
      live[u] = q < nq && kk < K;
      if (live[u]) {
        ca[u] = load_codes<BITS>(a.q + rowA * pitch + (int64_t)kk * BITS / 8);
        cb[u] = load_codes<BITS>(a.q + rowB * pitch + (int64_t)kk * BITS / 8);
        const int b = kk / p.block;
        sa[u] = scale_half2(__ldg(a.s + rowA * nblk + b), p.dtype);
        sb[u] = scale_half2(__ldg(a.s + rowB * nblk + b), p.dtype);
        za[u] = zp_half2(a.zp, rowA * nblk + b, BITS);
        zb[u] = zp_half2(a.zp, rowB * nblk + b, BITS);
      }
    }
#pragma unroll
    for (int u = 0; u < kChunksPerBatch; ++u) {
      const int q = q0 + u * a.ksplit;
      if (q >= nq) break;
      uint32_t pa[16], pb[16];
      if (live[u]) {
        dequant_pairs<BITS>(ca[u], za[u], sa[u], pa);
        dequant_pairs<BITS>(cb[u], zb[u], sb[u], pb);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pa[i] = pb[i] = 0u;
      }
      const uint4* xq = xs + q * 128;
      uint32_t bw[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = xq[i * 32 + lane];
        bw[4 * i] = v.x; bw[4 * i + 1] = v.y; bw[4 * i + 2] = v.z; bw[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma16816(acc, pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1], bw[2 * s], bw[2 * s + 1]);
    }
  }

  // fixed-order reduction of the split-K partial tiles
  if (warp < a.ksplit) {
#pragma unroll
    for (int r = 0; r < 4; ++r) red[(warp * 32 + lane) * 4 + r] = acc[r];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    const int L = threadIdx.x >> 2, r = threadIdx.x & 3;
    float v = 0.f;
    for (int w = 0; w < a.ksplit; ++w) v += red[(w * 32 + L) * 4 + r];
    const int gg = L >> 2, cc = L & 3;
    const int row = gg + ((r & 2) ? 8 : 0);
    const int n = 2 * cc + (r & 1);
    tile[row * 8 + n] = v;
  }
  __syncthreads();

  if constexpr (FC1) {
    if (threadIdx.x < 64) {
      const int j = threadIdx.x >> 3, n = threadIdx.x & 7;
      if (n < n_e) {
        const int pos = begin + n;
        const int t = ws.sorted_route[pos] / p.k;
        const float sigma = ws.tok_scale[t];
        const float inv = 1.0f / sigma;
        const float gt = tile[(2 * j) * 8 + n] * inv;
        const float ut = tile[(2 * j + 1) * 8 + n] * inv;
        const float h = silu(gt) * ut * sigma * sigma;
        const int jg = row0 / 2 + j;
        ws.h16[(int64_t)pos * p.I + permuted_pos(jg, perm_group(p.bits))] =
            __half_as_ushort(__float2half_rn(h));
      }
    }
  } else {
    if (threadIdx.x < 128) {
      const int row = threadIdx.x & 15, n = threadIdx.x >> 4;
      if (n < n_e) {
        const int pos = begin + n;
        const int r = ws.sorted_route[pos];
        const int t = r / p.k;
        const float inv = 1.0f / ws.tok_scale[t];
        ws.y[(int64_t)r * p.H + row0 + row] = tile[row * 8 + n] * inv * inv * ws.topk_w[r];
      }
    }
  }
}

template <int BITS, bool FC1>
cudaError_t launch_one(const DecodeArgs& a, int active_max, cudaStream_t s) {
  const int nq = (a.K + kChunkK - 1) / kChunkK;
  const size_t smem = (size_t)nq * 4 * 32 * 16 + (size_t)a.ksplit * 32 * 4 * 4 + 16 * 8 * 4;
  if (smem > 48 * 1024) {
    const cudaError_t err = cudaFuncSetAttribute(decode_gemv_kernel<BITS, FC1>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  dim3 grid(a.N / kRowsPerCta, active_max);
  const int warps = a.ksplit > 4 ? a.ksplit : 4;  // >= 128 threads for the epilogue
  decode_gemv_kernel<BITS, FC1><<<grid, 32 * warps, smem, s>>>(a);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_bits(const Problem& p, bool fc1, const uint8_t* q, const void* scales,
                        const uint8_t* zp, const Workspace& ws, cudaStream_t s) {
  const int64_t R = p.R();
  const int active_max = (int)(R < p.E ? R : p.E);
  DecodeArgs a{q, static_cast<const uint16_t*>(scales), zp, fc1 ? ws.x16 : ws.h16,
               fc1 ? 2 * p.I : p.H, fc1 ? p.H : p.I, 0, p, ws};
  const int nq = (a.K + kChunkK - 1) / kChunkK;
  a.ksplit = nq < kMaxKsplit ? nq : kMaxKsplit;
  return fc1 ? launch_one<BITS, true>(a, active_max, s) : launch_one<BITS, false>(a, active_max, s);
}

}  // namespace

cudaError_t launch_decode(const Problem& p, bool fc1, const uint8_t* q, const void* scales,
                          const uint8_t* zp, const Workspace& ws, cudaStream_t s) {
  switch (p.bits) {
    case 4: return launch_bits<4>(p, fc1, q, scales, zp, ws, s);
    case 3: return launch_bits<3>(p, fc1, q, scales, zp, ws, s);
    case 2: return launch_bits<2>(p, fc1, q, scales, zp, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qmoe
