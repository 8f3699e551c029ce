// grouped.cu -- grouped per-expert dequant-GEMM path on tcgen05 (sm_103a).
//
// For T > 8 the routes are grouped by expert (sorted order) and cut into tiles
// of 256 consecutive sorted rows that all belong to one expert, the grouped
// prefill scheme of the pages (BuildInt3ExpertTilesKernel / sorted expert map
// feeding the grouped GEMMs, "[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload
// ..." #33731; CUTLASS MoeFCGemm for INT4 prefill). A persistent CTA per SM walks
// its share of (256-row tile, BN-column tile) works and computes D = A * W_e^T:
//
//   warp 0       code producer: per K stage the packed code tile of W_e and,
//                every 8 scale blocks, a box of block scales (or, with zero
//                points, it loads the stage's scales and zero points itself);
//   warp 22      activation producer: per K stage the A tile (FP16
//                activations, 128B-swizzled);
//                both by cp.async.bulk.tensor into rings of shared-memory slots
//                with mbarrier transaction counts;
//   warp 1       allocates TMEM; one lane issues tcgen05.mma (kind::f16, two
//                M = 128 accumulators sharing each B stage, N = BN, K = 16) and
//                commits each stage's A and B slots back to their writers;
//   warps 2..17  dequantise the code tile to FP16 ((code - zp) * s, exact for
//                BF16 scales) into the 128B-swizzled K-major B layout, in two
//                groups of 8 warps that take alternate stages;
//   warps 18..21 after each tile, read the accumulators (tcgen05.ld) and run
//                the epilogue while warps 2..17 work on the next tile; with
//                128-row weight tiles (INT3) the accumulators are double
//                buffered and the MMAs of the next tile run meanwhile too.
//
// Operands are FP16 (not BF16): (code - zp) * scale needs up to 11 significant
// bits, which FP16 holds exactly and BF16 does not; FP16 and BF16 run at the
// same tensor rate. fc1 epilogue: SwiGLU of the interleaved gate/up columns,
// FP16 store in the K-order permutation of the fc2 operand. fc2 epilogue: FP32
// rows scaled by the routing weight, stored per route id for the combine.
//
// Weights-stationary works (WS; few routes per expert, e.g. a mid-size batch):
// tiles of at most 128 sorted rows of one expert, and the operands trade
// places. The dequantised tile of 128 weight rows is the MMA's A (M = 128) and
// the tile's routes are B, N = the routes rounded up to 16, copied in boxes of
// 16 rows; D holds weight rows on the TMEM lanes and routes on the columns. An
// expert with a handful of routes then pays for 16-route MMA columns instead of
// a 128-row route tile, the activation ring is a quarter the size, and the code
// ring is deep enough to keep the weight stream in flight.
//
// Every mbarrier wait gives up after a bounded time: the CTA then records an
// error code in the workspace, drains its copies and MMAs in flight, frees its
// TMEM and returns.
#include "tma.cuh"
#include <cuda_fp8.h>

namespace qmoe {
namespace {

constexpr int kSubM = 128;             // rows per MMA / TMEM accumulator
constexpr int kBM = 2 * kSubM;         // rows per tile: two accumulators share each B stage
constexpr int kGroupWarps = 8;         // one dequantisation group
constexpr int kDequantWarps = 2 * kGroupWarps;   // warps 2..17: two groups taking alternate stages
constexpr int kDequantThreads = 32 * kGroupWarps;  // threads of one group (one stage)
constexpr int kEpiWarps = 4;           // warps 18..21: one per TMEM lane quarter
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kAProdWarp = 2 + kDequantWarps + kEpiWarps;   // warp 22
constexpr int kThreads = 32 * (kAProdWarp + 1);
constexpr uint64_t kWaitLimitNs = QMOE_WAIT_LIMIT_NS;
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 0.1 s
constexpr int kErrTimeout = 1;
static_assert(kBM == kTileM, "the grouping kernels cut tiles of kTileM sorted rows");

// TSC: block scales brought in by bulk tensor copies (no zero points, and rows of
// scales a multiple of 16 bytes): one [BN rows][8 scales] box covers 8 blocks
// along K (a "scale span" of 8*block/BK stages) in a ring of two; otherwise the
// producer warp loads scales and zero points per stage and stores FP16 words.
// WS: the weights-stationary form (see the top of the file).
template <int BITS, bool TSC, bool FC1, bool WS>
struct Cfg {
  // K per stage. INT3 takes 128 (a 32-code unit of INT3 is 12 bytes; a code copy
  // must be a multiple of 16 bytes per row).
  static constexpr int BK = BITS == 3 ? 128 : 64;
  // Weight rows per tile (MMA N; WS: M, as two 128-row halves). With 128 (INT3
  // route tiles), a tile's two accumulators take 256 TMEM columns, so two tiles'
  // accumulators fit (ACC = 2) and the epilogue of one tile overlaps the MMAs of
  // the next. INT4 / INT2 keep 256 and one accumulator buffer: 128 there
  // (double-buffered) measured slower for fc2, as every activation tile then
  // feeds half as many MMAs. WS: the same rows, as 128-row halves (M = 128 each)
  // with accumulators of up to 128 route columns, double-buffered; every stage's
  // fixed cost (its barrier hand-offs) is spread over 256 rows for INT4 / INT2,
  // which measured worth more than the deeper rings 128 rows would leave room
  // for.
  static constexpr int BN = BITS == 3 ? 128 : 256;
  static constexpr int HALVES = BN / kSubM;           // WS: accumulators per tile
  static constexpr int AROWS = WS ? kTileWs : kBM;    // activation rows per stage
  static constexpr int ACC = WS ? 2 : (4 * BN <= 512 ? 2 : 1);   // accumulator buffers
  // Three rings: activation tiles (read by the MMAs), code tiles (read by the
  // dequantisers) and dequantised B tiles (written by the dequantisers, read by
  // the MMAs). The B ring only spans dequantisation to MMA; the two rings fed by
  // copies are deeper, so that more copies are in flight per SM. WS: the small
  // activation tiles leave room for a code ring of 8 (INT3) or 12 stages.
  static constexpr int SA = BITS == 3 ? 2 : 3;
  static constexpr int SC = WS ? (BITS == 3 ? 4 : 2) : (BITS == 3 ? 2 : (BITS == 4 ? 3 : 4));
  static constexpr int SB = BITS == 3 ? 2 : 3;
  static constexpr int SUB = BK / 64;                 // 64-wide swizzle atoms per stage
  // K per code copy. A weight row's codes are read in pieces of CK * BITS / 8
  // bytes; WS copies 256 K at once (128 bytes of INT4, 96 of INT3, 64 of INT2 per
  // row), which the dequantisers take as R = CK / BK stages, both groups sharing
  // each copy. (Each expert's weights there come from DRAM once; pieces of 32
  // bytes per row, spread over a whole tile's time, held its weight stream to a
  // fraction of the bandwidth.) Route tiles re-read each weight tile from L2 and
  // keep one copy per stage.
  static constexpr int CK = WS ? kWsCodeK : BK;
  static constexpr int R = CK / BK;
  static constexpr int A_BYTES = AROWS * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int CODE_ROW = BK * BITS / 8;      // bytes of codes per weight row per stage
  static constexpr int CODE_ROW_C = CK * BITS / 8;    // bytes per weight row per code copy
  static constexpr int C_BYTES = BN * CODE_ROW_C;
  static constexpr int UNIT_BYTES = 4 * BITS;         // 32 codes
  static constexpr int UNITS_PER_ROW = BK / 32;
  static constexpr int UNITS = BN * UNITS_PER_ROW;
  static constexpr int UNITS_PER_THREAD = UNITS / kDequantThreads;
  static constexpr int S_BYTES = UNITS * 4;           // per unit: FP16 scale | zero point << 16
  static constexpr int SC_BYTES = BN * 16;            // one scale box: [BN][8] 16-bit scales
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + SA * A_BYTES;
  static constexpr int C_OFF = B_OFF + SB * B_BYTES;
  static constexpr int S_OFF = C_OFF + SC * C_BYTES;
  static constexpr int BAR_OFF = S_OFF + (TSC ? 2 * SC_BYTES : SC * R * S_BYTES);
  static constexpr int NBARS = 2 * (SA + SC + SB) + 2 * ACC + 4;
  static constexpr int BAR_BYTES = WS ? 512 : 256;    // barriers, TMEM address, flags, fill words
  static constexpr int SMEM = BAR_OFF + BAR_BYTES + 1024;   // + alignment slack
  static_assert(8 * NBARS + 8 + 4 * SC <= BAR_BYTES, "barrier area");
  // two accumulators per tile; WS: one per 128 weight rows, of kTileWs columns
  static constexpr int TMEM_COLS = WS ? ACC * HALVES * kTileWs : 2 * BN * ACC;
  static_assert(UNITS % kDequantThreads == 0, "units must split evenly");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// ------------------------------------------------------------------ PTX wrappers

// Bounded wait that ignores the abort flags (used to drain work in flight).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > kDrainLimitNs) return false;
  }
}

// Bounded wait. Returns false if this CTA or another CTA of the launch gave up,
// or if the phase does not complete within kWaitLimitNs; in the last case the
// CTA's abort flag and the launch-wide error flag in the workspace are set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          volatile int* launch_err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 255u) == 0 || kWaitLimitNs == 0) {
      if (*launch_err) {
        *abort_flag = 1;
        return false;
      }
      if (globaltimer_ns() - t0 >= kWaitLimitNs) {
        *abort_flag = 1;
        *launch_err = kErrTimeout;
        return false;
      }
    }
  }
}

// Bounded wait until a shared word equals `want`, with mbar_wait's abort rules.
__device__ __forceinline__ bool word_wait(const volatile int* word, int want, volatile int* abort_flag,
                                          volatile int* launch_err) {
  if (*word == want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (*word == want) return true;
    if (*abort_flag) return false;
    if ((i & 255u) == 0 || kWaitLimitNs == 0) {
      if (*launch_err) {
        *abort_flag = 1;
        return false;
      }
      if (globaltimer_ns() - t0 >= kWaitLimitNs) {
        *abort_flag = 1;
        *launch_err = kErrTimeout;
        return false;
      }
    }
  }
}

// 32-byte global store (one full sector), 32-byte aligned address.
__device__ __forceinline__ void st_global_v8(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t e, uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
               "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8 rows x 128 bytes per swizzle atom, atoms 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                          // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                          // swizzle mode: 128B
  return d;
}

// Instruction descriptor, kind::f16: FP32 accumulator, FP16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
        "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
        "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// ------------------------------------------------------------------ dequantisation

__device__ __forceinline__ uint32_t h2_sub_mul(uint32_t biased, uint32_t zp2, uint32_t s2) {
  const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&biased),
                                    *reinterpret_cast<const __half2*>(&zp2)),
                            *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The 16 FP16 pairs of 32 packed codes in the activations' K-order permutation
// (pair p holds stored K positions 2p and 2p+1; see perm_group).
template <int BITS>
__device__ __forceinline__ void dequant_unit(const uint32_t* w, uint32_t z2, uint32_t s2, uint32_t* pr) {
  constexpr uint32_t kMagic = 0x64006400u;  // FP16 1024.0 in both halves
  if constexpr (BITS == 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m)
        pr[4 * i + m] = h2_sub_mul(((w[i] >> (4 * m)) & 0x000F000Fu) | kMagic, z2, s2);
  } else if constexpr (BITS == 2) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int m = 0; m < 8; ++m)
        pr[8 * i + m] = h2_sub_mul(((w[i] >> (2 * m)) & 0x00030003u) | kMagic, z2, s2);
  } else {
    const uint32_t v0 = __byte_perm(w[0], w[1], 0x4310), v1 = __byte_perm(w[0], w[1], 0x5421);
    const uint32_t v2 = __byte_perm(w[1], w[2], 0x6532), v3 = __byte_perm(w[1], w[2], 0x7643);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint32_t lo = m < 5 ? (v0 >> (3 * m)) : (v1 >> (3 * m - 8));
      const uint32_t hi = m < 5 ? (v2 >> (3 * m)) : (v3 >> (3 * m - 8));
      pr[m] = h2_sub_mul((lo & 0x00070007u) | kMagic, z2, s2);
      pr[8 + m] = h2_sub_mul((hi & 0x00070007u) | kMagic, z2, s2);
    }
  }
}


// FP4 formats (see qmoe.h): byte r of w (codes 2r and 2r + 1) as an FP16 pair,
// low half from the low nibble (the hardware conversion; exact). The FP4
// activations are in natural K order, so pair p is codes 2p and 2p + 1.
__device__ __forceinline__ uint32_t e2m1x2(uint32_t w, int r) {
  const uint32_t b = (w >> (8 * r)) & 0xFFu;
  uint32_t h;
  asm("{\n .reg .b8 q;\n cvt.u8.u32 q, %1;\n cvt.rn.f16x2.e2m1x2 %0, q;\n}\n" : "=r"(h) : "r"(b));
  return h;
}

// FP16 bits of an FP4 block scale: E8M0 relative to 2^ref (the epilogue applies
// 2^ref in FP32), or E4M3 as it is (exact in FP16).
__device__ __forceinline__ uint16_t fp4_scale_bits(int fmt, uint32_t b, int ref) {
  if (fmt == QMOE_FORMAT_MXFP4) {
    if (b == 0xFFu) return (uint16_t)0x7E00u;
    const int e16 = (int)b - 127 - ref + 15;     // FP16 exponent field of 2^(b - 127 - ref)
    if (e16 >= 1 && e16 <= 30) return (uint16_t)(e16 << 10);
    return __half_as_ushort(__float2half_rn(ldexpf(1.0f, (int)b - 127 - ref)));
  }
  return __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3).x;
}

// MXFP4: the exponent of the first E8M0 scale of expert e's matrix (N rows).
__device__ __forceinline__ int mx_ref(const void* scales, int e, int N, int nblk) {
  const uint8_t b = __ldg(static_cast<const uint8_t*>(scales) + (int64_t)e * N * nblk);
  return b == 0xFF ? 0 : min(max((int)b - 127, -100), 100);
}

__device__ __forceinline__ int permuted_pos(int j, int G) {
  const int base = j - j % G, i = j % G;
  return base + (i < G / 2 ? 2 * i : 2 * (i - G / 2) + 1);
}

struct GemmArgs {
  const uint16_t* scales;  // [E][N][K/block]
  const uint8_t* zp;       // [E][N][K/block] or null
  int N, K;
  Problem p;
  Workspace ws;
};

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 v = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 32 codes -> 16 FP16 pairs in the activations' K-order permutation. INT4 uses
// the in-place nibble decode (bits 4-7 read as 1024 + 16c and rescaled exactly by
// one FMA with 1/16); INT2/INT3 cut each pair with a shift and a mask.
template <int BITS>
__device__ __forceinline__ void dequant_unit_fast(const uint32_t* w, uint32_t zp, uint32_t s2, uint32_t* pr) {
  constexpr uint32_t kMagic = 0x64006400u;
  const uint32_t z1 = (0x6400u + zp) * 0x00010001u;  // 1024 + zp
  if constexpr (BITS == 4) {
    // -(64 + zp), exactly representable for zp in 0..15
    const __half2 nz = __float2half2_rn(-(64.0f + (float)zp));
    const uint32_t z16v = *reinterpret_cast<const uint32_t*>(&nz);
    constexpr uint32_t kSixteenth = 0x2C002C00u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = w[i], v8 = w[i] >> 8;
      pr[4 * i + 0] = h2_mul(h2_sub(lop3_and_or(v, 0x000F000Fu, kMagic), z1), s2);
      pr[4 * i + 1] = h2_mul(h2_fma(lop3_and_or(v, 0x00F000F0u, kMagic), kSixteenth, z16v), s2);
      pr[4 * i + 2] = h2_mul(h2_sub(lop3_and_or(v8, 0x000F000Fu, kMagic), z1), s2);
      pr[4 * i + 3] = h2_mul(h2_fma(lop3_and_or(v8, 0x00F000F0u, kMagic), kSixteenth, z16v), s2);
    }
  } else {
    dequant_unit<BITS>(w, z1, s2, pr);
  }
}


template <int BITS, bool FC1, bool TSC, bool WS>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_s, GemmArgs g) {
  pdl_wait();
  pdl_trigger();
  using C = Cfg<BITS, TSC, FC1, WS>;
  constexpr int SA = C::SA, SB = C::SB, SC = C::SC;
  const Workspace& ws = g.ws;
  const Problem& p = g.p;
  volatile int* launch_err = ws.counters + 2;   // set by a CTA whose wait timed out
  const int K = g.K, N = g.N;
  const int ksteps = K / C::BK;
  const int n_tiles_n = (N + C::BN - 1) / C::BN;
  // work tiles, m-tile major so that the n-tiles of one activation tile run together
  const int works = ws.counters[1] * n_tiles_n;
  if (blockIdx.x >= works || *launch_err) return;
  const int my_works = (works - blockIdx.x + gridDim.x - 1) / gridDim.x;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  // activation ring: landed / read by the MMAs; code ring: landed (with the
  // stage's scales) / read by the dequantisers; B ring: dequantised / read by the
  // MMAs; then accumulators ready / drained by the epilogue, and the scale-box
  // ring (TSC): box landed / box read by the dequantisers
  auto bar_afull = [&](int s) { return bar0 + 8u * s; };
  auto bar_aempty = [&](int s) { return bar0 + 8u * (SA + s); };
  auto bar_cfull = [&](int s) { return bar0 + 8u * (2 * SA + s); };
  auto bar_cempty = [&](int s) { return bar0 + 8u * (2 * SA + SC + s); };
  auto bar_bready = [&](int s) { return bar0 + 8u * (2 * SA + 2 * SC + s); };
  auto bar_bempty = [&](int s) { return bar0 + 8u * (2 * SA + 2 * SC + SB + s); };
  constexpr int kAcc = 2 * (SA + SC + SB);
  auto bar_accum = [&](int b) { return bar0 + 8u * (kAcc + b); };
  auto bar_drained = [&](int b) { return bar0 + 8u * (kAcc + C::ACC + b); };
  auto bar_sfull = [&](int b) { return bar0 + 8u * (kAcc + 2 * C::ACC + b); };
  auto bar_sempty = [&](int b) { return bar0 + 8u * (kAcc + 2 * C::ACC + 2 + b); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::BAR_OFF + 8 * C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBARS + 4);
  // per code slot: the stage whose copy the producer issued into it last
  volatile int* cfill = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(bar_afull(s), 1);                 // the copy issue (with its byte count)
      mbar_init(bar_aempty(s), 1);                // MMA commit
    }
    for (int s = 0; s < SC; ++s) {
      mbar_init(bar_cfull(s), TSC ? 1 : 1 + 32);  // the copy issue [+ 32 scale writers]
      mbar_init(bar_cempty(s), kDequantThreads * C::R);   // every stage of the copy
      cfill[s] = -1;
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bar_bready(s), kDequantThreads);
      mbar_init(bar_bempty(s), 1);                // MMA commit
    }
    for (int b = 0; b < C::ACC; ++b) {
      mbar_init(bar_accum(b), 1);
      mbar_init(bar_drained(b), kEpiThreads);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_sfull(b), 1);
      mbar_init(bar_sempty(b), 2 * kDequantThreads);   // both groups (a group alone arrives twice)
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
    if (TSC) asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_s)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32((const void*)tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nblk = K / p.block;
  const int span = 8 * p.block / C::BK;          // stages per scale box (TSC)
  const int kcopies = ksteps / C::R;             // code copies per tile (K is a multiple of CK)
  auto tile_of = [&](int j, int& e, int& row0, int& n0) {
    const int w = blockIdx.x + j * gridDim.x;
    const int mt = w / n_tiles_n;
    e = ws.tiles[2 * mt];
    row0 = ws.tiles[2 * mt + 1];
    n0 = (w - mt * n_tiles_n) * C::BN;
  };
  // 128-row halves of a tile that hold routes (1 or 2): an expert's last tile
  // often fills only the first, and its second half is neither copied nor
  // multiplied nor stored
  auto halves_of = [&](int e, int row0) { return ws.offsets[e + 1] - row0 > kSubM ? 2 : 1; };

  if (warp == 0) {
    // ---------------- code producer: per code copy (R stages) the code tile (lane 0)
    // and either a scale box every `span` stages (lane 0) or the stages' scales
    // (all lanes)
    int issued = 0, spans = 0;
    bool go = true;
    for (int j = 0; j < my_works && go; ++j) {
      int e, row0, n0;
      tile_of(j, e, row0, n0);
      const int64_t wrow_base = (int64_t)e * N + n0;
      const int64_t wrow_end = (int64_t)p.E * N;
      for (int ci = 0; ci < kcopies; ++ci) {
        const int ic = j * kcopies + ci;         // copy sequence number across tiles
        const int s = ic % SC;
        const uint32_t ph = (uint32_t)(ic / SC) & 1u;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(bar_cempty(s), ph ^ 1u, abort_flag, launch_err) ? 1 : 0;
        if constexpr (TSC) {
          // the scale boxes of the copy's stages that start a span, into the ring
          // slot the dequantisers released
#pragma unroll
          for (int sub = 0; sub < C::R; ++sub) {
            const int i = ci * C::R + sub;
            if (i % span != 0) continue;
            const int m = spans++;
            if (lane == 0 && ok) {
              if (m >= 2 && !mbar_wait(bar_sempty(m & 1), (uint32_t)((m - 2) >> 1) & 1u, abort_flag, launch_err))
                ok = 0;
              else {
                mbar_expect_tx(bar_sfull(m & 1), C::SC_BYTES);
                tma_load_2d(sbase + C::S_OFF + (m & 1) * C::SC_BYTES, &tmap_s, bar_sfull(m & 1),
                            i * C::BK / p.block, e * N + n0);
              }
            }
          }
        }
        if (__shfl_sync(0xffffffffu, ok, 0) == 0) { go = false; break; }
        ++issued;
        if (lane == 0) {
          cfill[s] = ic;
          mbar_expect_tx(bar_cfull(s), C::C_BYTES);
          tma_load_2d(sbase + C::C_OFF + s * C::C_BYTES, &tmap_q, bar_cfull(s), ci * C::CODE_ROW_C, e * N + n0);
        }
        if constexpr (TSC) continue;
#pragma unroll 1
        for (int sub = 0; sub < C::R; ++sub) {
          const int k0 = (ci * C::R + sub) * C::BK;
          uint32_t* st = reinterpret_cast<uint32_t*>(smem + C::S_OFF + (s * C::R + sub) * C::S_BYTES);
          // per batch of 8: all loads first (independent, no branches), then convert and store
          constexpr int PER_LANE = C::UNITS / 32;
          constexpr int BATCH = PER_LANE < 8 ? PER_LANE : 8;
          static_assert(PER_LANE % BATCH == 0, "scale batches");
          if (BITS == 4 && p.format != QMOE_FORMAT_INT) {
            // FP4: the 8-bit scales of each unit of 32 codes (one E8M0, or two E4M3 for
            // the 16-wide NVFP4 blocks) as two FP16 words, the first 16 codes' low
            const uint8_t* s8 = reinterpret_cast<const uint8_t*>(g.scales);
            const bool nv = p.format == QMOE_FORMAT_NVFP4;
#pragma unroll 1
            for (int q0 = 0; q0 < PER_LANE; q0 += BATCH) {
              // the batch's loads first (independent), then convert and store
              uint32_t b0[BATCH], b1[BATCH];
#pragma unroll
              for (int q = 0; q < BATCH; ++q) {
                const int u = lane + 32 * (q0 + q);
                const int r = u / C::UNITS_PER_ROW, jj = u % C::UNITS_PER_ROW;
                const int64_t wr = min(wrow_base + r, wrow_end - 1);
                const int64_t idx = wr * nblk + (k0 + 32 * jj) / p.block;
                b0[q] = __ldg(s8 + idx);
                b1[q] = nv ? __ldg(s8 + idx + 1) : 0u;
              }
#pragma unroll
              for (int q = 0; q < BATCH; ++q) {
                const int u = lane + 32 * (q0 + q);
                const int r = u / C::UNITS_PER_ROW;
                // the raw scale bytes; the dequantisers convert them (rows past the
                // array: a zero E4M3 / the smallest E8M0 with no rows to scale)
                st[u] = wrow_base + r < wrow_end ? (b0[q] | ((nv ? b1[q] : b0[q]) << 8)) : 0u;
              }
            }
            continue;
          }
#pragma unroll 1
          for (int q0 = 0; q0 < PER_LANE; q0 += BATCH) {
            uint16_t sv[BATCH];
            uint8_t zv[BATCH];
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
              const int u = lane + 32 * (q0 + q);
              const int r = u / C::UNITS_PER_ROW, jj = u % C::UNITS_PER_ROW;
              const int64_t wr = min(wrow_base + r, wrow_end - 1);   // rows past the array: masked below
              const int64_t idx = wr * nblk + (k0 + 32 * jj) / p.block;
              sv[q] = __ldg(g.scales + idx);
              zv[q] = g.zp ? __ldg(g.zp + idx) : (uint8_t)(1u << (BITS - 1));
            }
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
              const int u = lane + 32 * (q0 + q);
              const int r = u / C::UNITS_PER_ROW;
              const uint16_t sh = p.dtype == QMOE_BF16
                                      ? __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)sv[q] << 16)))
                                      : sv[q];
              st[u] = wrow_base + r < wrow_end ? ((uint32_t)sh | ((uint32_t)zv[q] << 16)) : 0u;
            }
          }
        }
        mbar_arrive(bar_cfull(s));
      }
    }
    if (lane == 0 && *abort_flag) {
      // let the copies already issued land before the CTA exits
      for (int i = issued - SC > 0 ? issued - SC : 0; i < issued; ++i)
        mbar_wait_drain(bar_cfull(i % SC), (uint32_t)(i / SC) & 1u);
      if (TSC)
        for (int m = spans - 2 > 0 ? spans - 2 : 0; m < spans; ++m)
          mbar_wait_drain(bar_sfull(m & 1), (uint32_t)(m >> 1) & 1u);
    }
  } else if (warp == kAProdWarp) {
    // ---------------- activation producer (lane 0): per stage the two 128-row halves
    // of the A tile
    if (lane == 0) {
      int issued = 0;
      bool go = true;
      for (int j = 0; j < my_works && go; ++j) {
        int e, row0, n0;
        tile_of(j, e, row0, n0);
        const int nh = WS ? 0 : halves_of(e, row0);
        // WS: the tile's routes in boxes of 16 rows (the MMA's N in steps of 16)
        const int nb = WS ? (min(kTileWs, ws.offsets[e + 1] - row0) + 15) / 16 : 0;
        for (int i = 0; i < ksteps; ++i) {
          const int it = j * ksteps + i;
          const int s = it % SA;
          const uint32_t ph = (uint32_t)(it / SA) & 1u;
          if (!mbar_wait(bar_aempty(s), ph ^ 1u, abort_flag, launch_err)) { go = false; break; }
          ++issued;
          const int k0 = i * C::BK;
          if constexpr (WS) {
            mbar_expect_tx(bar_afull(s), (uint32_t)(C::SUB * nb * 2048));
#pragma unroll
            for (int sub = 0; sub < C::SUB; ++sub)
              for (int b = 0; b < nb; ++b)
                tma_load_2d(sbase + C::A_OFF + s * C::A_BYTES + sub * (C::AROWS * 128) + b * 2048, &tmap_a,
                            bar_afull(s), k0 + 64 * sub, row0 + 16 * b);
          } else {
            mbar_expect_tx(bar_afull(s), (uint32_t)(C::A_BYTES / 2 * nh));
#pragma unroll
            for (int sub = 0; sub < C::SUB; ++sub)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if (h < nh)
                  tma_load_2d(sbase + C::A_OFF + s * C::A_BYTES + sub * (kBM * 128) + h * (kSubM * 128), &tmap_a,
                              bar_afull(s), k0 + 64 * sub, row0 + h * kSubM);
          }
        }
      }
      if (*abort_flag)
        for (int i = issued - SA > 0 ? issued - SA : 0; i < issued; ++i)
          mbar_wait_drain(bar_afull(i % SA), (uint32_t)(i / SA) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: two 128-row accumulators share each B stage
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kSubM, C::BN);
      bool go = true;
      int commits0 = 0, commits1 = 0;            // accumulator commits per buffer
      int buf = 0;
      bool pending = false;                      // MMAs issued since the last accumulator commit
      for (int j = 0; j < my_works && go; ++j) {
        buf = j % C::ACC;
        // the epilogue has read this buffer's previous tile
        if (j >= C::ACC &&
            !mbar_wait(bar_drained(buf), (uint32_t)(j / C::ACC - 1) & 1u, abort_flag, launch_err))
          break;
        tc_fence_after();
        const uint32_t acc0 = tmem + (uint32_t)(WS ? buf * C::HALVES * kTileWs : buf * 2 * C::BN);
        int e_t, row0_t, n0_t;
        tile_of(j, e_t, row0_t, n0_t);
        const int nh = WS ? 0 : halves_of(e_t, row0_t);
        // WS: M = the 128 dequantised weight rows, N = the tile's routes rounded up to 16
        const uint32_t idesc_ws =
            WS ? idesc_f16(kSubM, 16 * ((min(kTileWs, ws.offsets[e_t + 1] - row0_t) + 15) / 16)) : 0u;
        for (int i = 0; i < ksteps; ++i) {
          const int it = j * ksteps + i;
          const int sa = it % SA, sb = it % SB;
          if (!mbar_wait(bar_afull(sa), (uint32_t)(it / SA) & 1u, abort_flag, launch_err) ||
              !mbar_wait(bar_bready(sb), (uint32_t)(it / SB) & 1u, abort_flag, launch_err)) { go = false; break; }
          tc_fence_after();
          // one descriptor per slot; the others add their byte offset / 16 to its
          // start-address field (offsets within 2^18 bytes of shared memory: no
          // carry out of the field), so that each MMA issues after two additions
          const uint64_t a0 = sw128_desc(sbase + C::A_OFF + sa * C::A_BYTES);
          const uint64_t b0 = sw128_desc(sbase + C::B_OFF + sb * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            const int sub = kk / 4, off = (kk % 4) * 32;
            const uint64_t bdesc = b0 + (uint64_t)((sub * (C::BN * 128) + off) >> 4);
            if constexpr (WS) {
              // each 128-row half of the weight tile against the same routes
              const uint64_t adesc = a0 + (uint64_t)((sub * (C::AROWS * 128) + off) >> 4);
#pragma unroll
              for (int h = 0; h < C::HALVES; ++h)
                tc_mma(acc0 + h * kTileWs, bdesc + (uint64_t)((h * (kSubM * 128)) >> 4), adesc, idesc_ws,
                       (i | kk) != 0);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if (h < nh)
                  tc_mma(acc0 + h * C::BN, a0 + (uint64_t)((sub * (kBM * 128) + h * (kSubM * 128) + off) >> 4), bdesc,
                         idesc, (i | kk) != 0);
            }
          }
          pending = true;
          tc_commit(bar_aempty(sa));
          tc_commit(bar_bempty(sb));
        }
        if (!go) break;
        tc_commit(bar_accum(buf));
        if (buf == 0) ++commits0; else ++commits1;
        pending = false;
      }
      // MMAs in flight finish before TMEM is freed
      if (*abort_flag) {
        if (pending) {
          tc_commit(bar_accum(buf));
          if (buf == 0) ++commits0; else ++commits1;
        }
        if (commits0 > 0) mbar_wait_drain(bar_accum(0), (uint32_t)(commits0 - 1) & 1u);
        if (commits1 > 0) mbar_wait_drain(bar_accum(1), (uint32_t)(commits1 - 1) & 1u);
      }
    }
  } else if (warp < 2 + kDequantWarps) {
    // ---------------- dequantisation (warps 2..17): every stage's code tile to FP16 B.
    // Two groups of 8 warps take alternate stages (group g the stages whose
    // sequence number is g mod 2), so that one group's waits overlap the other's work.
    const int grp = (warp - 2) / kGroupWarps;
    const int t = threadIdx.x - 64 - grp * kDequantThreads;
    bool go = true;
    int box_seen = -1;                           // last scale box waited for (TSC)
    const int nbox = (ksteps + span - 1) / span; // scale boxes per tile (TSC)
    const uint32_t zdef = (uint32_t)(1u << (BITS - 1)) << 16;
    for (int j = 0; j < my_works && go; ++j) {
      // MXFP4: the tile's expert's reference exponent (its E8M0 scales become FP16 relative to it)
      int fref = 0;
      if (BITS == 4 && !TSC && p.format == QMOE_FORMAT_MXFP4) {
        int e, row0, n0;
        tile_of(j, e, row0, n0);
        fref = mx_ref(g.scales, e, N, nblk);
      }
      for (int i = 0; i < ksteps; ++i) {
        const int it = j * ksteps + i;
        if ((it & 1) != grp) continue;
        const int sub = i % C::R;                // stage within its code copy
        const int ic = j * kcopies + i / C::R;   // the copy's sequence number
        const int cs = ic % SC, bs = it % SB;
        // With one stage per copy and an odd ring the slot's previous copy belongs
        // to the other group. A parity wait would also pass while that copy is
        // still open, so wait first until the producer has issued this copy into
        // the slot: it does so only after the previous one was read, i.e. after it
        // landed. With R >= 2 (even) both groups read every copy, so each has seen
        // the slot's previous phase complete.
        if (C::R == 1 && SC % 2 == 1 && !word_wait(cfill + cs, ic, abort_flag, launch_err)) { go = false; break; }
        if (!mbar_wait(bar_cfull(cs), (uint32_t)(ic / SC) & 1u, abort_flag, launch_err)) { go = false; break; }
        const int m_cur = j * nbox + i / span;   // scale box of this stage (TSC), in issue order
        if (TSC && m_cur != box_seen) {
          box_seen = m_cur;
          if (!mbar_wait(bar_sfull(m_cur & 1), (uint32_t)(m_cur >> 1) & 1u, abort_flag, launch_err)) {
            go = false;
            break;
          }
        }
        // the MMAs have finished reading this B slot's previous stage
        if (!mbar_wait(bar_bempty(bs), ((uint32_t)(it / SB) & 1u) ^ 1u, abort_flag, launch_err)) {
          go = false;
          break;
        }
        // [BN rows][8] scales of this box; this stage's first block within it
        const uint16_t* sbox = reinterpret_cast<const uint16_t*>(smem + C::S_OFF + (m_cur & 1) * C::SC_BYTES);
        const int b_first = (i % span) * C::BK / p.block;
        const uint8_t* codes = smem + C::C_OFF + cs * C::C_BYTES + sub * C::CODE_ROW;
        const uint32_t* st = reinterpret_cast<const uint32_t*>(smem + C::S_OFF + (cs * C::R + sub) * C::S_BYTES);
        uint8_t* bt = smem + C::B_OFF + bs * C::B_BYTES;
#pragma unroll
        for (int u = 0; u < C::UNITS_PER_THREAD; ++u) {
          const int unit = t + kDequantThreads * u;
          const int r = unit / C::UNITS_PER_ROW, jj = unit % C::UNITS_PER_ROW;
          const uint8_t* src = codes + r * C::CODE_ROW_C + jj * C::UNIT_BYTES;
          uint32_t w[BITS];
          if constexpr (BITS == 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(src);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
          } else if constexpr (BITS == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(src);
            w[0] = v.x; w[1] = v.y;
          } else {
#pragma unroll
            for (int q = 0; q < 3; ++q) w[q] = reinterpret_cast<const uint32_t*>(src)[q];
          }
          uint32_t sz;
          if constexpr (TSC) {
            const uint16_t sb16 = sbox[r * 8 + b_first + (32 * jj) / p.block];
            const uint16_t sh = p.dtype == QMOE_BF16
                                    ? __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)sb16 << 16)))
                                    : sb16;
            sz = (uint32_t)sh | zdef;
          } else {
            sz = st[unit];
          }
          const uint32_t s2 = (sz & 0xFFFFu) * 0x00010001u;
          uint32_t pr[16];
          if (BITS == 4 && p.format != QMOE_FORMAT_INT) {
            // FP4: E2M1 pairs (natural order) times the scale of their 16 codes
            const uint32_t sa = fp4_scale_bits(p.format, sz & 0xFFu, fref) * 0x00010001u;
            const uint32_t sb2 = fp4_scale_bits(p.format, (sz >> 8) & 0xFFu, fref) * 0x00010001u;
#pragma unroll
            for (int q = 0; q < 16; ++q) pr[q] = h2_mul(e2m1x2(w[q >> 2], q & 3), q < 8 ? sa : sb2);
          } else {
            dequant_unit_fast<BITS>(w, sz >> 16, s2, pr);
          }
          uint8_t* rowp = bt + (jj >> 1) * (C::BN * 128) + r * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int chunk = (jj & 1) * 4 + c;
            *reinterpret_cast<uint4*>(rowp + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(pr[4 * c], pr[4 * c + 1], pr[4 * c + 2], pr[4 * c + 3]);
          }
        }
        fence_proxy_async();
        mbar_arrive(bar_bready(bs));
        mbar_arrive(bar_cempty(cs));
        // a group's last stage in a scale box releases the box for the group; a box
        // of one stage has one group, which arrives for both
        if (TSC) {
          const int box0 = (i / span) * span;
          const int box_end = min(box0 + span, ksteps);
          if (i + 2 >= box_end) mbar_arrive_cnt(bar_sempty(m_cur & 1), box_end - box0 >= 2 ? 1u : 2u);
        }
      }
    }
  } else if constexpr (WS) {
    // ---------------- epilogue (warps 18..21), weights-stationary: in accumulator
    // h (of C::HALVES), TMEM lane 32 (w % 4) + lane holds weight row f = n0 +
    // 128 h + 32 (w % 4) + lane of the tile, column c its route row0 + c. Each route's
    // factors are loaded by one lane and handed to the others by shuffles.
    const int quarter = warp & 3;
    for (int j = 0; j < my_works; ++j) {
      int e, row0, n0;
      tile_of(j, e, row0, n0);
      const int nr = min(kTileWs, ws.offsets[e + 1] - row0);
      const int f0 = n0 + quarter * 32 + lane;   // this thread's weight row in half 0
      // FP4: the factor the FP16 operands left out (MXFP4 2^ref, NVFP4 global scale)
      float ef = 1.0f;
      if constexpr (BITS == 4) {
        if (p.format == QMOE_FORMAT_MXFP4) ef = ldexpf(1.0f, mx_ref(g.scales, e, N, g.K / p.block));
        if (p.format == QMOE_FORMAT_NVFP4 && (FC1 ? p.g1 : p.g2)) ef = __ldg((FC1 ? p.g1 : p.g2) + e);
      }
      const float hn = h_norm(p, e);
      float2 bq[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      if (FC1 && p.b1)
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h)
          if (f0 + kSubM * h < N) bq[h] = fc1_bias_pair(p, e, (f0 + kSubM * h) >> 1);
      const int buf = j % C::ACC;
      if (!mbar_wait(bar_accum(buf), (uint32_t)(j / C::ACC) & 1u, abort_flag, launch_err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * C::HALVES * kTileWs);
      for (int c0 = 0; c0 < nr; c0 += 32) {
        const int c = c0 + lane;
        const bool ok = c < nr;
        const int rid_l = ok ? ws.sorted_route[row0 + c] : 0;
        const float sig_l = ok ? ws.tok_scale[rid_l / p.k] : 1.0f;
        const float inv1_l = 1.0f / sig_l;
        const float inv_l = ef * inv1_l;
#pragma unroll 1
        for (int h = 0; h < C::HALVES; ++h) {
          const int f = f0 + kSubM * h;
          uint32_t v[32];
          tmem_ld32(tbase + (uint32_t)(kTileWs * h + c0), v);
          if constexpr (FC1) {
            // rows 2m (gate) and 2m + 1 (up) of SwiGLU unit f / 2 sit in lanes 2m and
            // 2m + 1: the even lane finishes routes c0 .. c0 + 15, the odd one the rest
            const float ss_l = sig_l * sig_l * hn;
            const bool odd = lane & 1;
            const int jj = f >> 1;
            constexpr int G = BITS == 4 ? 8 : 16;
            const int col = (BITS == 4 && p.format != QMOE_FORMAT_INT) ? jj : permuted_pos(jj, G);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[16 + i], 1);
              const int cc = odd ? 16 + i : i;
              const float inv = __shfl_sync(0xffffffffu, inv_l, cc);
              const float ss = __shfl_sync(0xffffffffu, ss_l, cc);
              // SwiGLU with CUDA's fast exp and divide; the result is rounded to FP16
              const float gt = __uint_as_float(odd ? got : v[i]) * inv + bq[h].x;
              const float ut = __uint_as_float(odd ? v[16 + i] : got) * inv + bq[h].y;
              if (c0 + cc < nr && f < N)
                ws.h16[(int64_t)(row0 + c0 + cc) * p.I + col] =
                    __half_as_ushort(__float2half_rn(__fdividef(gt, 1.0f + __expf(-gt)) * ut * ss));
            }
          } else {
            const float fct_l = ok ? inv_l * inv1_l / hn * ws.topk_w[rid_l] : 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int rid = __shfl_sync(0xffffffffu, rid_l, i);
              const float fct = __shfl_sync(0xffffffffu, fct_l, i);
              if (c0 + i < nr && f < N) ws.y[(int64_t)rid * p.H + f] = __uint_as_float(v[i]) * fct;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_drained(buf));             // the accumulators may be overwritten
    }
  } else {
    // ---------------- epilogue (warps 18..21): warp w reads TMEM lanes 32 (w % 4) ..
    // of both accumulators, i.e. tile rows q*32 + lane and 128 + q*32 + lane, while
    // the dequantisers already work on the next tile's stages
    const int quarter = warp & 3;
    const int cpart = (warp - 2 - kDequantWarps) >> 2;   // with 4k epilogue warps: chunks cpart, cpart + k, ...
    for (int j = 0; j < my_works; ++j) {
      int e, row0, n0;
      tile_of(j, e, row0, n0);
      const int rows = min(kBM, ws.offsets[e + 1] - row0);
      int rid_h[2];
      float sigma_h[2], wr_h[2];
      bool ok_h[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int m = half * kSubM + quarter * 32 + lane;
        ok_h[half] = m < rows;
        rid_h[half] = ok_h[half] ? ws.sorted_route[row0 + m] : 0;
        sigma_h[half] = ok_h[half] ? ws.tok_scale[rid_h[half] / p.k] : 1.0f;
        wr_h[half] = FC1 ? 0.f : (ok_h[half] ? ws.topk_w[rid_h[half]] : 0.f);
      }
      // fc1 biases of the tile's BN weight rows, loaded before the accumulators are
      // waited for: lane l holds rows n0 + 8 l .. + 7 (four gate/up pairs); the
      // column loop takes its 16 pairs from the lanes by shuffles
      uint4 bias_v = make_uint4(0u, 0u, 0u, 0u);
      if (FC1 && p.b1 && 8 * lane < C::BN && n0 + 8 * lane < N)
        bias_v = __ldg(reinterpret_cast<const uint4*>(p.b1 + (int64_t)e * N + n0 + 8 * lane));
      const int buf = j % C::ACC;
      if (!mbar_wait(bar_accum(buf), (uint32_t)(j / C::ACC) & 1u, abort_flag, launch_err)) break;
      tc_fence_after();
      const int nh = rows > kSubM ? 2 : 1;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
      if (half >= nh) break;                     // no routes in this half (the same for the warp)
      const int pos = row0 + half * kSubM + quarter * 32 + lane;
      const int rid = rid_h[half];
      const float sigma = sigma_h[half], wr = wr_h[half];
      const bool row_ok = ok_h[half];
      const uint32_t tbase =
          tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * 2 * C::BN + half * C::BN);
      // FP4: the factor the FP16 operands left out (MXFP4 2^ref, NVFP4 global scale)
      float ef = 1.0f;
      if constexpr (BITS == 4) {
        if (p.format == QMOE_FORMAT_MXFP4) ef = ldexpf(1.0f, mx_ref(g.scales, e, N, g.K / p.block));
        if (p.format == QMOE_FORMAT_NVFP4 && (FC1 ? p.g1 : p.g2)) ef = __ldg((FC1 ? p.g1 : p.g2) + e);
      }
      const float inv1 = 1.0f / sigma;
      const float inv = ef * inv1;
      const float hn = h_norm(p, e);
      for (int c0 = 32 * cpart; c0 < C::BN; c0 += 32 * (kEpiWarps / 4)) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)c0, v);
        if (n0 + c0 >= N) continue;              // the same for the whole warp
        if constexpr (FC1) {
          // every lane takes part in the bias shuffles; rows past the tile's routes
          // (row_ok false) compute and store nothing
          // columns are W1 rows n0 + c0 .. +31: gate/up pairs -> 16 outputs h_j
          const int j0 = (n0 + c0) / 2;
          constexpr int G = BITS == 4 ? 8 : 16;
          const float ss = sigma * sigma * hn;
          uint16_t hv[16];
          // SwiGLU with CUDA's fast exp and divide; the result is rounded to FP16
          if (p.b1) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              // pair j0 + q = the tile's pair c0 / 2 + q: lane c0 / 8 + q / 4, element q % 4
              const uint32_t src = (q & 3) == 0 ? bias_v.x : (q & 3) == 1 ? bias_v.y : (q & 3) == 2 ? bias_v.z : bias_v.w;
              const uint32_t braw = __shfl_sync(0xffffffffu, src, (c0 >> 3) + (q >> 2));
              const float2 bq = make_float2(half_bits_to_float((uint16_t)(braw & 0xFFFFu), p.dtype),
                                            half_bits_to_float((uint16_t)(braw >> 16), p.dtype));
              const float gt = __uint_as_float(v[2 * q]) * inv + bq.x;
              const float ut = __uint_as_float(v[2 * q + 1]) * inv + bq.y;
              hv[q] = __half_as_ushort(__float2half_rn(__fdividef(gt, 1.0f + __expf(-gt)) * ut * ss));
            }
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float gt = __uint_as_float(v[2 * q]) * inv;
              const float ut = __uint_as_float(v[2 * q + 1]) * inv;
              hv[q] = __half_as_ushort(__float2half_rn(__fdividef(gt, 1.0f + __expf(-gt)) * ut * ss));
            }
          }
          uint16_t ov[16];
          if (BITS == 4 && p.format != QMOE_FORMAT_INT) {
#pragma unroll
            for (int q = 0; q < 16; ++q) ov[q] = hv[q];     // FP4: natural K order
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) ov[permuted_pos(q, G)] = hv[q];
          }
          // one 32-byte store: a whole sector per lane
          if (row_ok)
          st_global_v8(ws.h16 + (int64_t)pos * p.I + j0,
                       ov[0] | ((uint32_t)ov[1] << 16), ov[2] | ((uint32_t)ov[3] << 16),
                       ov[4] | ((uint32_t)ov[5] << 16), ov[6] | ((uint32_t)ov[7] << 16),
                       ov[8] | ((uint32_t)ov[9] << 16), ov[10] | ((uint32_t)ov[11] << 16),
                       ov[12] | ((uint32_t)ov[13] << 16), ov[14] | ((uint32_t)ov[15] << 16));
        } else {
          if (!row_ok) continue;
          const float f = inv * inv1 / hn * wr;
          float* dst = ws.y + (int64_t)rid * p.H + n0 + c0;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_global_v8(dst + 8 * q, __float_as_uint(__uint_as_float(v[8 * q]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 1]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 2]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 3]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 4]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 5]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 6]) * f),
                         __float_as_uint(__uint_as_float(v[8 * q + 7]) * f));
        }
      }
      }
      tc_fence_before();
      mbar_arrive(bar_drained(buf));             // the accumulators may be overwritten
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side

template <int BITS, bool FC1, bool TSC, bool WS>
cudaError_t launch_gemm_t(const Problem& p, const uint8_t* q, const void* scales, const uint8_t* zp,
                          const Workspace& ws, cudaStream_t s) {
  using C = Cfg<BITS, TSC, FC1, WS>;
  const int N = FC1 ? 2 * p.I : p.H;
  const int K = FC1 ? p.H : p.I;
  const int64_t R = p.R();
  const uint16_t* A = FC1 ? ws.x16s : ws.h16;
  CUtensorMap ta, tq, tsc;
  // activation boxes: 64 K x 128 rows (a route tile's half), WS 64 K x 16 routes
  if (!make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, (uint64_t)K, (uint64_t)R, (uint64_t)K * 2,
                   64, WS ? 16 : kSubM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t row_bytes = (uint64_t)K * BITS / 8;
  if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, row_bytes, (uint64_t)p.E * N, row_bytes,
                   C::CODE_ROW_C, C::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (TSC) {
    // [E*N rows][K/block] 16-bit scales, boxes of 8 scales x BN rows
    const uint64_t nb = (uint64_t)K / p.block;
    if (!make_map_2d(&tsc, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, nb, (uint64_t)p.E * N, nb * 2, 8, C::BN,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    tsc = tq;                                    // not read
  }
  const cudaError_t err = ensure_smem_optin(grouped_gemm_kernel<BITS, FC1, TSC, WS>, C::SMEM);
  if (err != cudaSuccess) return err;
  GemmArgs g{static_cast<const uint16_t*>(scales), zp, N, K, p, ws};
  // persistent: one CTA per SM, each walking its share of the (m-tile, n-tile) list
  const int sms = device_sm_count();
  const int64_t works_max = ws.max_tiles * ((N + C::BN - 1) / C::BN);
  dim3 grid((unsigned)(works_max < sms ? works_max : sms));
  return launch_pdl(grouped_gemm_kernel<BITS, FC1, TSC, WS>, grid, dim3(kThreads), C::SMEM, s, ta, tq, tsc, g);
}

// Scales by bulk tensor copies when there are no zero points and a row of
// scales is a multiple of 16 bytes; the producer-warp path otherwise. The
// weights-stationary kernel where the routing step cut tiles of kTileWs rows.
template <int BITS, bool FC1>
cudaError_t launch_gemm(const Problem& p, const uint8_t* q, const void* scales, const uint8_t* zp,
                        const Workspace& ws, cudaStream_t s) {
  const int K = FC1 ? p.H : p.I;
  const bool tsc = !zp && p.format == QMOE_FORMAT_INT && (K / p.block) % 8 == 0;
  if (p.tile_m == kTileWs)
    return tsc ? launch_gemm_t<BITS, FC1, true, true>(p, q, scales, zp, ws, s)
               : launch_gemm_t<BITS, FC1, false, true>(p, q, scales, zp, ws, s);
  if (p.tile_m != kTileM) return cudaErrorInvalidValue;
  return tsc ? launch_gemm_t<BITS, FC1, true, false>(p, q, scales, zp, ws, s)
             : launch_gemm_t<BITS, FC1, false, false>(p, q, scales, zp, ws, s);
}

}  // namespace

cudaError_t launch_grouped(const Problem& p, bool fc1, const uint8_t* q, const void* scales,
                           const uint8_t* zp, const Workspace& ws, cudaStream_t s) {
  switch (p.bits) {
    case 4: return fc1 ? launch_gemm<4, true>(p, q, scales, zp, ws, s) : launch_gemm<4, false>(p, q, scales, zp, ws, s);
    case 3: return fc1 ? launch_gemm<3, true>(p, q, scales, zp, ws, s) : launch_gemm<3, false>(p, q, scales, zp, ws, s);
    case 2: return fc1 ? launch_gemm<2, true>(p, q, scales, zp, ws, s) : launch_gemm<2, false>(p, q, scales, zp, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qmoe
