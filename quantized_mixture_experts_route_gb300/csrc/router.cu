// router.cu -- router logits ahead of routing: logits = x . W_router^T (sm_103a).
//
// The pages' RouterGateUpProj op runs one GEMM of the packed tokens with the
// router weight (together with a gate/up projection, outside this layer) and
// feeds its output to QMoE as raw logits ("[CUDA] Enable Tensor-Core INT3/INT4
// QMoE offload ..." #33731, "Vectorized SplitActivationVec8Kernel" item and the
// RouterGateUpProj per-row-count table). Here: x [T][H] and W_router [E][H] in
// the layer's dtype (BF16 or FP16), products on the tensor core (m16n8k16
// mma.sync with BF16 or FP16 operands as given, FP32 accumulation), each logit
// rounded once to the dtype (round to nearest even, NaN kept).
//
// Batches of up to 64 tokens: a block of 16 warps computes 8 experts for one
// tile of 16 tokens; the warps take consecutive K slices, each issuing the
// loads of eight K steps before their MMAs, and their FP32 partial sums are
// added in slice order in shared memory, so the result does not depend on
// timing. The router weight (E x H x 2 bytes) streams through E / 8 blocks.
// Larger batches: the tiled GEMM below (router_gemm_kernel).
#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

constexpr int kRWarps = 16;
constexpr int kRThreads = 32 * kRWarps;

template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t ld_pair(const uint16_t* row, int k, bool ok) {
  return ok ? __ldg(reinterpret_cast<const unsigned int*>(row + k)) : 0u;
}

template <bool BF16, int KS, int NF>
__global__ void __launch_bounds__(kRThreads) router_logits_kernel(Problem p, const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ w,
                                                                  uint16_t* __restrict__ logits) {
  constexpr int kRExperts = 8 * NF;    // experts per block: NF N-fragments
  // x may be the previous kernel's output (the previous layer)
  pdl_wait();
  pdl_trigger();
  constexpr int kTiles = kRWarps / KS;   // token tiles per block
  __shared__ float part[KS > 1 ? kRWarps : 1][NF][4][32];   // [warp][n-fragment][element][lane]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int slice = warp % KS, tile = warp / KS;
  const int64_t t0 = ((int64_t)blockIdx.y * kTiles + tile) * 16;
  const int e0 = blockIdx.x * kRExperts;
  const int H = p.H, E = p.E;
  const int nsteps = H / 16;
  const int s0 = nsteps * slice / KS, s1 = nsteps * (slice + 1) / KS;

  const bool r0 = t0 + g < p.T, r1 = t0 + g + 8 < p.T;
  const uint16_t* xa = x + (r0 ? (t0 + g) * H : 0);
  const uint16_t* xb = x + (r1 ? (t0 + g + 8) * H : 0);
  const uint16_t* wr[NF];
  bool ev[NF];
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const int e = e0 + f * 8 + g;
    ev[f] = e < E;
    wr[f] = w + (ev[f] ? (int64_t)e * H : 0);
  }
  float acc[NF][4];
#pragma unroll
  for (int f = 0; f < NF; ++f)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[f][i] = 0.f;

  // eight K steps per round, their loads issued before the MMAs
  for (int st0 = s0; st0 < s1; st0 += 8) {
    uint32_t a[8][4], b[8][NF][2];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = st0 + u < s1;
      const int k = (st0 + u) * 16 + 2 * c;
      a[u][0] = ld_pair(xa, k, in && r0);
      a[u][1] = ld_pair(xb, k, in && r1);
      a[u][2] = ld_pair(xa, k + 8, in && r0);
      a[u][3] = ld_pair(xb, k + 8, in && r1);
#pragma unroll
      for (int f = 0; f < NF; ++f) {
        b[u][f][0] = ld_pair(wr[f], k, in && ev[f]);
        b[u][f][1] = ld_pair(wr[f], k + 8, in && ev[f]);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int f = 0; f < NF; ++f)
        mma_16816<BF16>(acc[f], a[u][0], a[u][1], a[u][2], a[u][3], b[u][f][0], b[u][f][1]);
  }

  if constexpr (KS > 1) {
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int i = 0; i < 4; ++i) part[warp][f][i][lane] = acc[f][i];
    __syncthreads();
    if (slice != 0) return;
    // the tile's slices in K order
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = part[warp][f][i][lane];
        for (int s = 1; s < KS; ++s) v += part[warp + s][f][i][lane];
        acc[f][i] = v;
      }
  }

  // D fragment: rows g and g + 8 (tokens), columns 2c and 2c + 1 (experts)
#pragma unroll
  for (int f = 0; f < NF; ++f)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t t = t0 + g + ((i & 2) ? 8 : 0);
      const int e = e0 + f * 8 + 2 * c + (i & 1);
      if (t < p.T && e < E) logits[t * E + e] = float_to_half_bits(acc[f][i], p.dtype);
    }
}

// ---------------------------------------------------------------------------
// Larger batches: a tiled GEMM. A block computes 32 or 64 tokens x 128 experts;
// K moves in steps of 64 through a 4-stage ring of shared-memory tiles filled by
// 16-byte asynchronous copies (rows past T or E are filled with zeros), and each
// of the 8 warps multiplies 16 or 32 tokens x 32 experts from fragments read
// with ldmatrix. Rows are padded to 144 bytes so that the eight 16-byte rows an
// ldmatrix phase reads fall in distinct bank groups. The block's time is the
// SM's mma.sync throughput over its K loop (about 2 TFLOP/s per SM); 128-wide K
// steps halved the steps but not the time (8K tokens 22.6 us, 32K slower with
// one block per SM).
constexpr int kGN = 128, kGK = 64, kGStages = 4, kGPitch = 72;   // pitch in 16-bit elements
constexpr int kGThreads = 256;

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool BF16, int MT>
__global__ void __launch_bounds__(kGThreads) router_gemm_kernel(Problem p, const uint16_t* __restrict__ x,
                                                                const uint16_t* __restrict__ w,
                                                                uint16_t* __restrict__ logits) {
  constexpr int kGM = 32 * MT;               // tokens per block: MT 16-token tiles per warp
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint16_t gsm[];
  auto sa = reinterpret_cast<uint16_t(*)[kGM][kGPitch]>(gsm);                                // [stage]
  auto sb = reinterpret_cast<uint16_t(*)[kGN][kGPitch]>(gsm + kGStages * kGM * kGPitch);   // [stage]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int wm = warp & 1, wn = warp >> 1;     // token half of the block, 32-expert quarter
  const int64_t t0 = (int64_t)blockIdx.x * kGM;
  const int e0 = blockIdx.y * kGN;
  const int H = p.H, E = p.E;
  const int nk = H / kGK;

  auto load = [&](int kt, int st) {
    const int k0 = kt * kGK;
#pragma unroll
    for (int i = 0; i < (kGM * 8 + kGThreads - 1) / kGThreads; ++i) {
      const int idx = threadIdx.x + i * kGThreads, r = idx >> 3, q = idx & 7;
      if (idx < kGM * 8) {
        const bool ok = t0 + r < p.T;
        cp_async16_zfill((uint32_t)__cvta_generic_to_shared(&sa[st][r][q * 8]),
                         x + (ok ? (t0 + r) * H + k0 + q * 8 : 0), ok);
      }
    }
#pragma unroll
    for (int i = 0; i < (kGN * 8) / kGThreads; ++i) {
      const int idx = threadIdx.x + i * kGThreads, r = idx >> 3, q = idx & 7;
      const bool ok = e0 + r < E;
      cp_async16_zfill((uint32_t)__cvta_generic_to_shared(&sb[st][r][q * 8]),
                       w + (ok ? (int64_t)(e0 + r) * H + k0 + q * 8 : 0), ok);
    }
  };

  float acc[MT][4][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int f = 0; f < 4; ++f)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][f][i] = 0.f;

#pragma unroll
  for (int st = 0; st < kGStages - 1; ++st) {
    if (st < nk) load(st, st);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  for (int kt = 0; kt < nk; ++kt) {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kGStages - 2) : "memory");
    __syncthreads();                          // the stage is visible; the one refilled next is read
    if (kt + kGStages - 1 < nk) load(kt + kGStages - 1, (kt + kGStages - 1) % kGStages);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    const int st = kt % kGStages;
#pragma unroll
    for (int ks = 0; ks < kGK / 16; ++ks) {
      uint32_t a[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        ldmatrix_x4((uint32_t)__cvta_generic_to_shared(
                        &sa[st][(wm * MT + m) * 16 + (lane & 15)][ks * 16 + (lane >> 4) * 8]),
                    a[m][0], a[m][1], a[m][2], a[m][3]);
#pragma unroll
      for (int fp = 0; fp < 2; ++fp) {
        uint32_t b0, b1, b2, b3;
        const int row = wn * 32 + fp * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldmatrix_x4((uint32_t)__cvta_generic_to_shared(&sb[st][row][ks * 16 + ((lane >> 3) & 1) * 8]),
                    b0, b1, b2, b3);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          mma_16816<BF16>(acc[m][2 * fp], a[m][0], a[m][1], a[m][2], a[m][3], b0, b1);
          mma_16816<BF16>(acc[m][2 * fp + 1], a[m][0], a[m][1], a[m][2], a[m][3], b2, b3);
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");

#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int f = 0; f < 4; ++f)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + (wm * MT + m) * 16 + g + ((i & 2) ? 8 : 0);
        const int e = e0 + wn * 32 + f * 8 + 2 * c + (i & 1);
        if (t < p.T && e < E) logits[t * E + e] = float_to_half_bits(acc[m][f][i], p.dtype);
      }
}

template <bool BF16, int MT>
cudaError_t launch_gemm(const Problem& p, const uint16_t* x, const uint16_t* w, uint16_t* out, cudaStream_t s) {
  constexpr int kGM = 32 * MT;
  const size_t smem = sizeof(uint16_t) * kGStages * (kGM + kGN) * kGPitch;
  const cudaError_t err = ensure_smem_optin(router_gemm_kernel<BF16, MT>, (int)smem);
  if (err != cudaSuccess) return err;
  const dim3 grid((unsigned)((p.T + kGM - 1) / kGM), (p.E + kGN - 1) / kGN);
  return launch_pdl(router_gemm_kernel<BF16, MT>, grid, dim3(kGThreads), smem, s, p, x, w, out);
}

template <bool BF16>
cudaError_t launch_dtype(const Problem& p, const uint16_t* x, const uint16_t* w, uint16_t* out, cudaStream_t s) {
  if (p.T <= 64 || p.H % kGK != 0) {
    // decode-sized batches (and hidden sizes the tiled GEMM's K steps do not
    // divide): 8 experts per block, K split 16 ways, so that the router weight
    // streams through E / 8 blocks of 16 warps
    constexpr int KS = 16;
    const int64_t tiles = (p.T + 15) / 16;
    const dim3 grid((p.E + 7) / 8, (unsigned)tiles);
    return launch_pdl(router_logits_kernel<BF16, KS, 1>, grid, dim3(kRThreads), 0, s, p, x, w, out);
  }
  // 64 tokens per block once that still fills most SMs: the router weight is
  // then read from L2 half as often
  if ((p.T + 63) / 64 * ((p.E + kGN - 1) / kGN) * 5 >= 4 * (int64_t)device_sm_count())
    return launch_gemm<BF16, 2>(p, x, w, out, s);
  return launch_gemm<BF16, 1>(p, x, w, out, s);
}

}  // namespace

cudaError_t launch_router_logits(const Problem& p, const void* x, const void* w_router, void* logits,
                                 cudaStream_t s) {
  const auto* xx = static_cast<const uint16_t*>(x);
  const auto* ww = static_cast<const uint16_t*>(w_router);
  auto* out = static_cast<uint16_t*>(logits);
  return p.dtype == QMOE_BF16 ? launch_dtype<true>(p, xx, ww, out, s) : launch_dtype<false>(p, xx, ww, out, s);
}

}  // namespace qmoe
