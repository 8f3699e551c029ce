// decode.cu -- decode path (T <= 8): split-K dequant-GEMV kernels (sm_103a).
//
// For each expert that received routes, the selected expert's packed weight
// rows are streamed from HBM once, dequantised in registers and multiplied with
// the <= 8 routed activation rows on the tensor core (m16n8k16 mma.sync). The
// pages' decode kernels (MoeGemvTcInt4Kernel, FusedFc1FastVecKernel /
// Fc2RouteFastVecKernel, "[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload ..."
// #33731) group <= 8 routes of one expert per CTA around an m16n8k16 step; here
// the decode table pairs the routes of each active expert, so one MMA column pair
// serves two routes and every weight byte is read exactly once per call.
//
// Three kernels, by format:
//   decode_int4_tma_kernel  INT4, block 32, H and I multiples of 256 (the decode
//       stack's format): units of 16 or 32 weight rows x 256-wide K chunks,
//       brought into per-warp shared-memory rings by bulk tensor copies; codes
//       placed in FP16 mantissas and block scales applied in FP32 after the MMA;
//       stream-K split of the (unit, chunk) range into equal pieces per warp.
//   decode_int4_bs_kernel   the same arithmetic for other INT4 block-32 shapes
//       (K a multiple of 128), fed by per-lane cp.async.
//   decode_gemv_kernel      INT2, INT3 and other block sizes: FP16 dequantised
//       weights ((code - zp) * scale, exact for BF16 scales in the FP16 normal
//       range), persistent teams of warps over (expert, 16-row group) items with
//       K cut into 8 fixed slices added left to right.
//
// fc1 epilogue: h_i = silu(gate_i) * up_i from the interleaved rows 2i / 2i+1
// (activation_type "swiglu", swiglu_fusion = 1), stored in FP16 with the
// token's power of two squared. fc2 epilogue: y = (W2 h) / scale^2 * w_route in
// FP32, stored per route id for the combine.
#include "tma.cuh"
#include <cuda_fp8.h>

namespace qmoe {
namespace {

constexpr int kRowsPerGroup = 16;  // rows of one MMA M-fragment
constexpr int kWarps = 8;
constexpr int kChunkK = 128;       // K covered by one quad of lanes per chunk
constexpr int kSlices = 8;         // fixed K slices (the largest K split)

// 32 codes of one weight row (one lane's share of a chunk) plus the FP16 pair
// constants of its block: 1024 + zero point, and the scale.
template <int BITS>
struct RowChunk {
  uint32_t w[BITS];
  uint32_t z2, s2;
};

__device__ __forceinline__ uint32_t scale_half2(uint16_t bits, int dtype) {
  uint16_t h = bits;
  if (dtype == QMOE_BF16) h = __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)bits << 16)));
  return (uint32_t)h | ((uint32_t)h << 16);
}

__device__ __forceinline__ uint32_t h2_sub_mul(uint32_t biased, uint32_t zp2, uint32_t s2) {
  const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&biased),
                                    *reinterpret_cast<const __half2*>(&zp2)),
                            *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Words from which the FP16 pairs are cut. INT4 and INT2: the packed words. INT3:
// byte permutes that put two 8-code groups' bits into the two 16-bit halves
// (groups G0 = bytes 0-2, G1 = 3-5, G2 = 6-8, G3 = 9-11).
template <int BITS>
struct PairWords {
  uint32_t v[BITS == 3 ? 4 : BITS];
};

template <int BITS>
__device__ __forceinline__ PairWords<BITS> pair_words(const RowChunk<BITS>& r) {
  PairWords<BITS> o;
  if constexpr (BITS == 3) {
    o.v[0] = __byte_perm(r.w[0], r.w[1], 0x4310);  // G0 bits 0-15  | G1 bits 0-15
    o.v[1] = __byte_perm(r.w[0], r.w[1], 0x5421);  // G0 bits 8-23  | G1 bits 8-23
    o.v[2] = __byte_perm(r.w[1], r.w[2], 0x6532);  // G2 bits 0-15  | G3 bits 0-15
    o.v[3] = __byte_perm(r.w[1], r.w[2], 0x7643);  // G2 bits 8-23  | G3 bits 8-23
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) o.v[i] = r.w[i];
  }
  return o;
}

// Dequantised FP16 pair p (0..15) of a lane's 32 codes, in the activations'
// K-order permutation: pair p holds stored K positions 2p and 2p+1.
template <int BITS>
__device__ __forceinline__ uint32_t dq_pair(const PairWords<BITS>& w, int p, uint32_t z2, uint32_t s2) {
  constexpr uint32_t kMagic = 0x64006400u;  // FP16 1024.0 in both halves
  uint32_t bits;
  if constexpr (BITS == 4) {
    bits = (w.v[p >> 2] >> (4 * (p & 3))) & 0x000F000Fu;   // codes (8i+m, 8i+m+4)
  } else if constexpr (BITS == 2) {
    bits = (w.v[p >> 3] >> (2 * (p & 7))) & 0x00030003u;   // codes (16i+m, 16i+m+8)
  } else {
    const int g = p >> 3, m = p & 7;                        // codes (16g+m, 16g+m+8)
    bits = m < 5 ? (w.v[2 * g] >> (3 * m)) & 0x00070007u : (w.v[2 * g + 1] >> (3 * m - 8)) & 0x00070007u;
  }
  return h2_sub_mul(bits | kMagic, z2, s2);
}

struct DecodeArgs {
  const uint8_t* q;        // [E][N][K*bits/8]
  const uint16_t* s;       // [E][N][K/block]
  const uint8_t* zp;       // [E][N][K/block] or null
  const uint16_t* act;     // FC1: x16 [T][K] by token; FC2: h16 [R][K] by sorted position
  int N, K;
  int ks;                  // warps per team (K split of one item), 1, 2, 4 or 8
  Problem p;
  Workspace ws;
  const float* gsc;        // NVFP4: per-expert FP32 global scales of this matmul, or null
};

// ---- FP4 expert formats (E2M1 codes, 8-bit block scales; see qmoe.h)
// Byte r of w (codes 2r and 2r + 1) as an FP16 pair, low half from the low
// nibble (the hardware conversion, exact: every E2M1 value is an FP16 value).
// The FP4 formats keep the activations in natural K order (kX16Natural), so
// the pairs are adjacent codes.
__device__ __forceinline__ uint32_t e2m1x2(uint32_t w, int r) {
  const uint32_t b = (w >> (8 * r)) & 0xFFu;
  uint32_t h;
  asm("{\n .reg .b8 q;\n cvt.u8.u32 q, %1;\n cvt.rn.f16x2.e2m1x2 %0, q;\n}\n" : "=r"(h) : "r"(b));
  return h;
}

// FP16 bits of a block scale: E8M0 times 2^-ref (ref: the expert's reference
// exponent, taken back in FP32 by the epilogue), or E4M3 as it is (exact in FP16).
template <int FMT>
__device__ __forceinline__ uint32_t fp4_scale_half(uint32_t b, int ref) {
  if constexpr (FMT == QMOE_FORMAT_MXFP4) {
    if (b == 0xFFu) return 0x7E00u;
    return __half_as_ushort(__float2half_rn(ldexpf(1.0f, (int)b - 127 - ref)));
  } else {
    return __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3).x;
  }
}

// Index of h_j in the permuted FP16 row layout.
__device__ __forceinline__ int permuted_pos(int j, int G) {
  const int base = j - j % G, i = j % G;
  return base + (i < G / 2 ? 2 * i : 2 * (i - G / 2) + 1);
}

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

// INT4: the 16 FP16 pairs of 32 codes. Nibbles at bits 0-3 become 1024 + c in the
// FP16 mantissa (one AND/OR); nibbles at bits 4-7 become 1024 + 16c, which one
// FMA by 1/16 turns into 64 + c exactly; a single shift by 8 serves the other
// two nibble positions. (c - zp) is exact, and so is (c - zp) * scale for BF16
// scales in the FP16 normal range.
__device__ __forceinline__ void dequant_int4(const uint32_t* w, uint32_t z1, uint32_t z16, uint32_t s2,
                                             uint32_t* pr) {
  constexpr uint32_t kMagic = 0x64006400u;     // 1024.0 | 1024.0
  constexpr uint32_t kSixteenth = 0x2C002C00u; // 0.0625 | 0.0625
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = w[i], v8 = w[i] >> 8;
    pr[4 * i + 0] = h2_mul(h2_sub(lop3_and_or(v, 0x000F000Fu, kMagic), z1), s2);
    pr[4 * i + 1] = h2_mul(h2_fma(lop3_and_or(v, 0x00F000F0u, kMagic), kSixteenth, z16), s2);
    pr[4 * i + 2] = h2_mul(h2_sub(lop3_and_or(v8, 0x000F000Fu, kMagic), z1), s2);
    pr[4 * i + 3] = h2_mul(h2_fma(lop3_and_or(v8, 0x00F000F0u, kMagic), kSixteenth, z16), s2);
  }
}

template <int BITS>
__device__ __forceinline__ void dequant_chunk(const RowChunk<BITS>& r, uint32_t* pr) {
  if constexpr (BITS == 4) {
    // z2 holds 1024 + zp; -(64 + zp) = -(z - 960) for the 1/16-scaled nibbles
    const __half2 z = *reinterpret_cast<const __half2*>(&r.z2);
    const __half2 z16h = __hneg2(__hsub2(z, __float2half2_rn(960.0f)));
    dequant_int4(r.w, r.z2, *reinterpret_cast<const uint32_t*>(&z16h), r.s2, pr);
  } else {
    const PairWords<BITS> pw = pair_words<BITS>(r);
#pragma unroll
    for (int q = 0; q < 16; ++q) pr[q] = dq_pair<BITS>(pw, q, r.z2, r.s2);
  }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Copy one lane's 32 codes of one row (4*BITS bytes) into its shared slot.
template <int BITS>
__device__ __forceinline__ void copy_codes(uint32_t dst, const uint8_t* src) {
  if constexpr (BITS == 4) {
    cp_async16(dst, src);
  } else if constexpr (BITS == 2) {
    cp_async8(dst, src);
  } else {
    cp_async4(dst, src);
    cp_async4(dst + 4, src + 4);
    cp_async4(dst + 8, src + 8);
  }
}

constexpr int kRing = 8;        // chunks in flight per warp (shared-memory ring)

// Per-item data of the decode table entry of one active expert.
struct ItemMeta {
  int e, begin, n_e, tok;       // tok: token of route slot g (this lane's activation row)
  int ref;                      // MXFP4: exponent of the expert's first block scale
  float hn;                     // the expert's SwiGLU normalisation (h_norm), read one item ahead
};

template <int BITS, bool FC1, int FMT>
__global__ void __launch_bounds__(32 * kWarps, 2) decode_gemv_kernel(DecodeArgs a) {
  pdl_wait();
  pdl_trigger();
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  const int K = a.K, N = a.N;
  const int nq = (K + kChunkK - 1) / kChunkK;
  const int rgroups = N / kRowsPerGroup;
  const int items = ws.counters[0] * rgroups;   // (expert's chunk of <= 8 routes, 16-row group) pairs

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ks = a.ks;
  const int team = warp / ks, ksi = warp % ks;
  const int teams_per_block = kWarps / ks;
  const int team_global = blockIdx.x * teams_per_block + team;
  const int teams_total = gridDim.x * teams_per_block;
  const int sl0 = kSlices * ksi / ks, sl1 = kSlices * (ksi + 1) / ks;
  const int cb = nq * sl0 / kSlices, ce = nq * sl1 / kSlices;
  const int cpi = ce - cb;                       // chunks per item for this warp (>= 1)
  const int my_items = team_global < items ? (items - team_global + teams_total - 1) / teams_total : 0;
  const int total = my_items * cpi;
  const int64_t pitch = (int64_t)K * BITS / 8;
  const int nblk = K / p.block;
  const int lb = 31 - __clz(p.block);
  constexpr int kChunkBytes = kChunkK * BITS / 8;
  const int chunk_scales = kChunkK >> lb;

  extern __shared__ __align__(16) uint8_t smem[];
  // per warp: [kRing][2 rows][32 lanes][16 B] of codes; then the split-K buffers
  const uint32_t ring_base = (uint32_t)__cvta_generic_to_shared(smem) + warp * (kRing * 2 * 32 * 16);
  // per warp, after the code rings: [kRing][32 lanes] scale words and zero-point words
  // (each lane reads back only what it wrote), then the split-K buffers
  uint32_t* const sring = reinterpret_cast<uint32_t*>(smem + kWarps * kRing * 2 * 32 * 16) + warp * (2 * kRing * 32);
  uint32_t* const zring = sring + kRing * 32;
  float* red = reinterpret_cast<float*>(smem + kWarps * kRing * 2 * 32 * 16 + kWarps * 2 * kRing * 32 * 4);
  float* tred = red + (size_t)team * kSlices * 32 * 4;

  auto meta_of = [&](int it) {
    ItemMeta m{0, 0, 0, 0, 0, 1.0f};
    if (it < items) {
      // the chunks of one expert are consecutive, so the items that read the same
      // weight rows run at about the same time and the repeats hit L2
      const int act = ws.active[it / rgroups];
      m.e = act & 0xFFFF;
      m.begin = ws.offsets[m.e] + (act >> 16) * kDecodeChunk;
      m.n_e = min(kDecodeChunk, ws.offsets[m.e + 1] - m.begin);
      m.tok = g < m.n_e ? ws.sorted_route[m.begin + g] / p.k : 0;
      m.hn = h_norm(p, m.e);
      if constexpr (FMT == QMOE_FORMAT_MXFP4) {
        // E8M0 block scales span 2^-127 .. 2^127: the FP16 operands carry them
        // relative to the expert's first one, whose power of two the epilogue applies
        const uint8_t b0 = __ldg(reinterpret_cast<const uint8_t*>(a.s) + (int64_t)m.e * N * (K / p.block));
        m.ref = b0 == 0xFF ? 0 : min(max((int)b0 - 127, -100), 100);
      }
    }
    return m;
  };

  // ---- issue side: code rows of (pf_item, pf_cc) -> ring slot; scales -> register ring
  int pf_item = team_global, pf_cc = 0;
  ItemMeta pf_next = meta_of(pf_item);
  const uint8_t* pq = nullptr;
  const uint16_t* ps = nullptr;
  const uint8_t* pz = nullptr;
  int64_t pso = 0;               // FP4 formats: element offset of the chunk's first 8-bit scale
  int pkk = 0;
  auto issue = [&](int slot_u) {
    if (pf_cc == 0) {
      const ItemMeta m = pf_next;
      pf_next = meta_of(pf_item + teams_total);
      const int slot = pf_item / rgroups;
      const int64_t row = (int64_t)m.e * N + (pf_item - slot * rgroups) * kRowsPerGroup + g;
      pkk = cb * kChunkK + 32 * c;
      pq = a.q + row * pitch + (int64_t)pkk * BITS / 8;
      ps = a.s + row * nblk + (pkk >> lb);
      pso = row * nblk + (pkk >> lb);
      pz = a.zp ? a.zp + row * nblk + (pkk >> lb) : nullptr;
    }
    const uint32_t dst = ring_base + slot_u * (2 * 32 * 16) + lane * 16;
    if (pkk < K) {
      copy_codes<BITS>(dst, pq);
      copy_codes<BITS>(dst + 32 * 16, pq + 8 * pitch);
      if constexpr (FMT == QMOE_FORMAT_INT) {
        sring[slot_u * 32 + lane] = (uint32_t)__ldg(ps) | ((uint32_t)__ldg(ps + 8 * nblk) << 16);
        zring[slot_u * 32 + lane] = pz ? ((uint32_t)__ldg(pz) | ((uint32_t)__ldg(pz + 8 * nblk) << 16))
                           : ((1u << (BITS - 1)) * 0x00010001u);
      } else {
        // 8-bit scales of rows g and g + 8: one each per 32 codes (MXFP4), two (NVFP4)
        const uint8_t* s8 = reinterpret_cast<const uint8_t*>(a.s) + pso;
        if constexpr (FMT == QMOE_FORMAT_MXFP4)
          sring[slot_u * 32 + lane] = (uint32_t)__ldg(s8) | ((uint32_t)__ldg(s8 + 8 * nblk) << 16);
        else
          sring[slot_u * 32 + lane] = (uint32_t)__ldg(s8) | ((uint32_t)__ldg(s8 + 1) << 8) |
                          ((uint32_t)__ldg(s8 + 8 * nblk) << 16) | ((uint32_t)__ldg(s8 + 8 * nblk + 1) << 24);
        zring[slot_u * 32 + lane] = 0u;
      }
    } else {
      sring[slot_u * 32 + lane] = 0u;   // zero scale: stale codes in the slot contribute exact zeros
      zring[slot_u * 32 + lane] = 0u;
    }
    cp_async_commit();
    pq += kChunkBytes;
    ps += chunk_scales;
    pso += chunk_scales;
    if (pz) pz += chunk_scales;
    pkk += kChunkK;
    if (++pf_cc == cpi) { pf_cc = 0; pf_item += teams_total; }
  };

#pragma unroll
  for (int u = 0; u < kRing - 1; ++u) {
    if (u < total) issue(u);
    else cp_async_commit();
  }

  // ---- compute side
  int item = team_global, cc = 0;
  ItemMeta cur = meta_of(item), nxt = meta_of(item + teams_total);
  auto brow_of = [&](const ItemMeta& m) -> const uint16_t* {
    if (g >= m.n_e) return nullptr;
    const int64_t row = FC1 ? (int64_t)m.tok : (int64_t)(m.begin + g);
    return a.act + row * K + cb * kChunkK + 32 * c;
  };
  const uint16_t* brow = brow_of(cur);
  uint32_t bnext[16];
  auto load_b = [&](const uint16_t* src, int q) {
    if (src != nullptr && q * kChunkK + 32 * c < K) {
      const uint4* v4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = __ldg(v4 + j);
        bnext[4 * j] = v.x; bnext[4 * j + 1] = v.y; bnext[4 * j + 2] = v.z; bnext[4 * j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) bnext[j] = 0u;
    }
  };
  if (total > 0) load_b(brow, cb);

  float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f}, tot[4] = {0.f, 0.f, 0.f, 0.f};
  int slice = sl0;
  int row0 = (item % (rgroups > 0 ? rgroups : 1)) * kRowsPerGroup;
  auto close_slices_until = [&](int gq) {
    while (slice < sl1 && nq * (slice + 1) / kSlices <= gq) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float v = acc0[r] + acc1[r];
        if (ks == 1)
          tot[r] = slice == 0 ? v : tot[r] + v;
        else
          tred[(slice * 32 + lane) * 4 + r] = v;
        acc0[r] = acc1[r] = 0.f;
      }
      ++slice;
    }
  };

  // one rolled loop over the warp's chunks (its body once in the instruction
  // stream: unrolled over the ring, the body with its epilogue overflowed the
  // instruction cache)
#pragma unroll 1
  for (int f = 0; f < total; ++f) {
    {
      const int u = f % kRing;
      // keep kRing chunks in flight: issue f + kRing - 1 into the slot freed last iteration
      if (f + kRing - 1 < total) issue((u + kRing - 1) % kRing);
      else cp_async_commit();
      cp_async_wait<kRing - 1>();   // chunk f has landed

      const int q = cb + cc;
      close_slices_until(q);
      uint32_t bw[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) bw[j] = bnext[j];
      // next chunk's activations (same item, or the next item's first chunk)
      if (cc + 1 < cpi) load_b(brow ? brow + (cc + 1) * kChunkK : nullptr, q + 1);
      else load_b(brow_of(nxt), cb);

      RowChunk<BITS> ra, rb;
      const uint8_t* slotp = smem + warp * (kRing * 2 * 32 * 16) + u * (2 * 32 * 16) + lane * 16;
      if constexpr (BITS == 4) {
        const uint4 va = *reinterpret_cast<const uint4*>(slotp);
        const uint4 vb = *reinterpret_cast<const uint4*>(slotp + 32 * 16);
        ra.w[0] = va.x; ra.w[1] = va.y; ra.w[2] = va.z; ra.w[3] = va.w;
        rb.w[0] = vb.x; rb.w[1] = vb.y; rb.w[2] = vb.z; rb.w[3] = vb.w;
      } else if constexpr (BITS == 2) {
        const uint2 va = *reinterpret_cast<const uint2*>(slotp);
        const uint2 vb = *reinterpret_cast<const uint2*>(slotp + 32 * 16);
        ra.w[0] = va.x; ra.w[1] = va.y;
        rb.w[0] = vb.x; rb.w[1] = vb.y;
      } else {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          ra.w[i] = reinterpret_cast<const uint32_t*>(slotp)[i];
          rb.w[i] = reinterpret_cast<const uint32_t*>(slotp + 32 * 16)[i];
        }
      }
      const uint32_t sp = sring[u * 32 + lane], zp2 = zring[u * 32 + lane];
      uint32_t pa[16], pb[16];
      if constexpr (FMT == QMOE_FORMAT_INT) {
        ra.s2 = scale_half2((uint16_t)(sp & 0xFFFFu), p.dtype);
        rb.s2 = scale_half2((uint16_t)(sp >> 16), p.dtype);
        ra.z2 = (0x6400u + (zp2 & 0xFFFFu)) * 0x00010001u;
        rb.z2 = (0x6400u + (zp2 >> 16)) * 0x00010001u;
        dequant_chunk<BITS>(ra, pa);
        dequant_chunk<BITS>(rb, pb);
      } else {
        // E2M1 pairs times the block scale: pair q holds codes 2q and 2q + 1 (byte
        // q % 4 of word q / 4), the first 16 codes (words 0, 1) in the first NVFP4 block
        uint32_t sa[2], sb[2];
        if constexpr (FMT == QMOE_FORMAT_MXFP4) {
          sa[0] = sa[1] = fp4_scale_half<FMT>(sp & 0xFFu, cur.ref) * 0x00010001u;
          sb[0] = sb[1] = fp4_scale_half<FMT>((sp >> 16) & 0xFFu, cur.ref) * 0x00010001u;
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            sa[h] = fp4_scale_half<FMT>((sp >> (8 * h)) & 0xFFu, 0) * 0x00010001u;
            sb[h] = fp4_scale_half<FMT>((sp >> (16 + 8 * h)) & 0xFFu, 0) * 0x00010001u;
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          pa[q] = h2_mul(e2m1x2(ra.w[q >> 2], q & 3), sa[q >> 3]);
          pb[q] = h2_mul(e2m1x2(rb.w[q >> 2], q & 3), sb[q >> 3]);
        }
      }
#pragma unroll
      for (int s = 0; s < 8; s += 2) {
        mma16816(acc0, pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1], bw[2 * s], bw[2 * s + 1]);
        mma16816(acc1, pa[2 * s + 2], pb[2 * s + 2], pa[2 * s + 3], pb[2 * s + 3], bw[2 * s + 2], bw[2 * s + 3]);
      }
      if (++cc < cpi) continue;

      // ---- item finished: close its slices, reduce split K in slice order, epilogue
      close_slices_until(nq);
      if (ks > 1) {
        asm volatile("bar.sync %0, %1;\n" ::"r"(team + 1), "r"(32 * ks) : "memory");
        if (ksi == 0) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float v = tred[lane * 4 + r];
            for (int sl = 1; sl < kSlices; ++sl) v += tred[(sl * 32 + lane) * 4 + r];
            tot[r] = v;
          }
        }
      }
      if (ksi == 0) {
        const int n0 = 2 * c, n1 = 2 * c + 1;
        const int begin = cur.begin, n_e = cur.n_e;
        if constexpr (FMT != QMOE_FORMAT_INT) {
          // the factor the FP16 operands left out: the MXFP4 reference power of
          // two, or the NVFP4 global scale of the expert's matrix
          const float ef = FMT == QMOE_FORMAT_MXFP4 ? ldexpf(1.0f, cur.ref) : (a.gsc ? __ldg(a.gsc + cur.e) : 1.0f);
#pragma unroll
          for (int r = 0; r < 4; ++r) tot[r] *= ef;
        }
        if constexpr (FC1) {
          // gate rows are even, up rows odd: lane g+1 (lane + 4) holds the up rows of lane g
          float up[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) up[r] = __shfl_down_sync(0xffffffffu, tot[r], 4);
          if ((g & 1) == 0) {
            const int G = perm_group(p.bits);
            const int j_lo = row0 / 2 + g / 2, j_hi = j_lo + 4;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int n = (r & 1) ? n1 : n0;
              if (n < n_e) {
                const float sigma = ws.tok_scale[ws.sorted_route[begin + n] / p.k];
                const float inv = 1.0f / sigma;
                const int j = (r & 2) ? j_hi : j_lo;
                const float2 bj = fc1_bias_pair(p, cur.e, j);
                const float h = silu(tot[r] * inv + bj.x) * (up[r] * inv + bj.y) * (sigma * sigma * cur.hn);
                const int pos = FMT == QMOE_FORMAT_INT ? permuted_pos(j, G) : j;   // FP4: natural order
                ws.h16[(int64_t)(begin + n) * p.I + pos] = __half_as_ushort(__float2half_rn(h));
              }
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int n = (r & 1) ? n1 : n0;
            if (n < n_e) {
              const int rid = ws.sorted_route[begin + n];
              const float inv = 1.0f / ws.tok_scale[rid / p.k];
              const int row = row0 + g + ((r & 2) ? 8 : 0);
              ws.y[(int64_t)rid * p.H + row] = tot[r] * (inv * inv / cur.hn) * ws.topk_w[rid];
            }
          }
        }
      }
      if (ks > 1) asm volatile("bar.sync %0, %1;\n" ::"r"(team + 1), "r"(32 * ks) : "memory");
      // next item
      cc = 0;
      item += teams_total;
      cur = nxt;
      nxt = meta_of(item + teams_total);
      brow = brow_of(cur);
      row0 = (item % rgroups) * kRowsPerGroup;
      slice = sl0;
#pragma unroll
      for (int r = 0; r < 4; ++r) acc0[r] = acc1[r] = 0.f;
    }
  }
  cp_async_wait<0>();
}

int sm_count();
int64_t decode_grid_blocks();
constexpr int kBlocksPerSm = 2;

// ---------------------------------------------------------------------------
// INT4, block 32: block scales applied after the MMA
//
// Per weight the kernel only places the code in an FP16 mantissa: (v & 0x000F000F)
// | 1024.0 gives 1024 + c for the nibbles at bits 0-3, and (v & 0x00F000F0) |
// 1024.0 gives 1024 + 16c for the nibbles at bits 4-7 (the odd K positions of the
// activations' layout). The activations carry 1/16 at odd K positions, so every
// product is (1024 + c) * x exactly. A second MMA per step with the constant
// operand -(1024 + zp) (even positions) / -(1024 + 16 zp) (odd positions) removes
// the bias and the zero point, leaving sum_k (c_k - zp) x_k in FP32.
//
// That sum must be taken per 32-wide block, since each block has its own scale:
// the B operand is laid out so that D column n = 4t + b only receives the K
// positions of block b of the chunk (lane c of a quad owns block c, and only the
// lanes with groupID % 4 == c supply a token's activations). The FP32 block sums
// are then scaled by their block's scale with one FMA each and accumulated per
// column; the four block columns of a token are added at the end. Two tokens
// share one MMA; larger expert batches take several.
// ---------------------------------------------------------------------------
constexpr int kRingB = 4;                          // chunks in flight per warp
constexpr int kSlotCode = 2 * 32 * 16;             // [2 rows][32 lanes][16 B]
constexpr int kSlotScale = 2 * 32 * 4;             // [2 rows][32 lanes][2 scales]
constexpr int kSlotZp = 2 * 32 * 4;                // [2 rows][32 lanes][4 zero points]
constexpr int kSlotAct = 8 * 64;                   // [8 owner lanes][32 activations]
constexpr int kSlotBytes = kSlotCode + kSlotScale + kSlotZp + kSlotAct;
constexpr int kBlocksPerSmB = 3;
constexpr int kMinPiece = 8;                       // chunks per warp at least (small batches)

// Stream-K work split. Units are (decode-table entry = active expert and a pair
// of its routes, 16-row group); their 128-wide K chunks, laid end to end, form
// one flat range that is cut into nw equal contiguous pieces, one per warp of a
// persistent grid. A warp streams its piece through the cp.async ring; a unit that
// lies wholly inside the piece ends in the warp's epilogue, and the (at most two)
// units cut at the piece's ends leave an FP32 partial tile in scratch and take a
// ticket: the last of a unit's parts adds them in chunk order (deterministic)
// and runs the epilogue. An expert with more than two routes has several
// entries whose units read the same weight rows; neighbouring entries stream at
// the same time, so the repeated reads are served by L2.
__device__ __forceinline__ int chunk_owner(int64_t x, int nw, int64_t total) {
  // the warp whose piece [floor(w*total/nw), floor((w+1)*total/nw)) holds chunk x
  return (int)(((x + 1) * nw - 1) / total);
}

template <bool FC1, bool BF16S, bool HAS_ZP>
__global__ void __launch_bounds__(32 * kWarps, kBlocksPerSmB) decode_int4_bs_kernel(DecodeArgs a) {
  pdl_wait();
  pdl_trigger();
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  const int K = a.K, N = a.N;
  const int nq = K / kChunkK;                    // K is a multiple of 128 here
  const int rgroups = N / kRowsPerGroup;
  const int items = ws.counters[3] * rgroups;
  const int64_t cfull = (int64_t)items * nq;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int wg = blockIdx.x * kWarps + warp;
  // pieces of at least kMinPiece chunks (and so never empty: the tickets count
  // one part per warp between a unit's first and last chunk)
  const int64_t nw_cap = (cfull + kMinPiece - 1) / kMinPiece;
  const int nw = (int)((int64_t)gridDim.x * kWarps < nw_cap ? (int64_t)gridDim.x * kWarps : nw_cap);
  const int64_t x_begin = wg < nw ? cfull * wg / nw : 0, x_end = wg < nw ? cfull * (wg + 1) / nw : 0;
  const int total = (int)(x_end - x_begin);
  const int64_t pitch = K / 2;                   // bytes of codes per row
  const int nblk = K / 32;
  const int b0 = 2 * (c & 1);                    // blocks of this lane's D columns: b0, b0 + 1
  const bool owner = (g & 3) == c;               // supplies activations for column g
  const int oid = (g >> 2) * 4 + c;              // owner slot in the activation area
  const int on = g >> 2;                         // owner lane's route within the pair

  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* ring = smem + warp * (kRingB * kSlotBytes);
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);

  const int item0 = total > 0 ? (int)(x_begin / nq) : 0;
  const int cic0 = total > 0 ? (int)(x_begin - (int64_t)item0 * nq) : 0;

  // ---- issue side: walks the piece kRingB - 1 chunks ahead
  int p_item = item0, p_cic = cic0;              // unit and chunk within it
  bool p_new = true;
  const uint8_t* pq = nullptr;
  const uint16_t* ps = nullptr;
  const uint8_t* pz = nullptr;
  int pboff = -1;
  auto issue = [&](int slot) {
    if (p_new) {
      p_new = false;
      const int4 d0 = __ldg(reinterpret_cast<const int4*>(ws.dtab + (p_item / rgroups) * kDtabInts));
      const int4 d1 = __ldg(reinterpret_cast<const int4*>(ws.dtab + (p_item / rgroups) * kDtabInts + 4));
      const int64_t row = (int64_t)d0.x * N + (p_item % rgroups) * kRowsPerGroup + g;
      pq = a.q + row * pitch + (p_cic * kChunkK + 32 * c) / 2;
      ps = a.s + row * nblk + p_cic * 4 + b0;
      if constexpr (HAS_ZP) pz = a.zp + row * nblk + p_cic * 4;
      pboff = -1;
      if (owner && on < d0.z) pboff = (FC1 ? (on ? d1.y : d1.x) : d0.y + on) * K + p_cic * kChunkK + 32 * c;
    }
    const uint32_t d = ring_s + slot * kSlotBytes;
    cp_async16(d + lane * 16, pq);
    cp_async16(d + 512 + lane * 16, pq + 8 * pitch);
    cp_async4(d + kSlotCode + lane * 4, ps);
    cp_async4(d + kSlotCode + 128 + lane * 4, ps + 8 * nblk);
    if constexpr (HAS_ZP) {
      cp_async4(d + kSlotCode + kSlotScale + lane * 4, pz);
      cp_async4(d + kSlotCode + kSlotScale + 128 + lane * 4, pz + 8 * nblk);
      pz += 4;
    }
    if (pboff >= 0) {
      const uint16_t* src = a.act + pboff;
      const uint32_t da = d + kSlotCode + kSlotScale + kSlotZp + oid * 16;   // [4][8 owners][16 B]
      cp_async16(da, src);
      cp_async16(da + 128, src + 8);
      cp_async16(da + 256, src + 16);
      cp_async16(da + 384, src + 24);
      pboff += kChunkK;
    }
    cp_async_commit();
    pq += kChunkK / 2;
    ps += 4;
    if (++p_cic == nq) { p_cic = 0; ++p_item; p_new = true; }
  };
  for (int u = 0; u < kRingB - 1; ++u) {
    if (u < total) issue(u);
    else cp_async_commit();
  }

  // constant operands removing the bias and the default zero point 8
  const __half2 ne_d = __float2half2_rn(-(1024.0f + 8.0f)), no_d = __float2half2_rn(-(1024.0f + 128.0f));
  const uint32_t ne_def = *reinterpret_cast<const uint32_t*>(&ne_d);
  const uint32_t no_def = *reinterpret_cast<const uint32_t*>(&no_d);

  // ---- compute side
  int item = item0, cic = cic0;
  int first_cic = cic;                           // where this warp's part of the unit began
  int cnt = 0, pos0 = 0, tok0 = 0, tok1 = 0;
  bool bvalid = false, fresh = true;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t bw[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) bw[j] = 0u;       // non-owner lanes keep zeros for good
  int slot = 0;
  for (int f = 0; f < total; ++f) {
    if (f + kRingB - 1 < total) issue((slot + kRingB - 1) % kRingB);
    else cp_async_commit();
    if (fresh) {
      fresh = false;
      const int4 d0 = __ldg(reinterpret_cast<const int4*>(ws.dtab + (item / rgroups) * kDtabInts));
      const int4 d1 = __ldg(reinterpret_cast<const int4*>(ws.dtab + (item / rgroups) * kDtabInts + 4));
      pos0 = d0.y;
      cnt = d0.z;
      tok0 = d1.x;
      tok1 = d1.y;
      bvalid = owner && on < cnt;
    }
    cp_async_wait<kRingB - 1>();
    const uint8_t* sl = ring + slot * kSlotBytes;
    const uint4 ca = *reinterpret_cast<const uint4*>(sl + lane * 16);
    const uint4 cbv = *reinterpret_cast<const uint4*>(sl + 512 + lane * 16);
    const uint32_t swa = *reinterpret_cast<const uint32_t*>(sl + kSlotCode + lane * 4);
    const uint32_t swb = *reinterpret_cast<const uint32_t*>(sl + kSlotCode + 128 + lane * 4);
    uint32_t ne_a = ne_def, ne_b = ne_def, no_a = no_def, no_b = no_def;
    if constexpr (HAS_ZP) {
      const uint32_t za = (*reinterpret_cast<const uint32_t*>(sl + kSlotCode + kSlotScale + lane * 4) >> (8 * c)) & 0xFFu;
      const uint32_t zb = (*reinterpret_cast<const uint32_t*>(sl + kSlotCode + kSlotScale + 128 + lane * 4) >> (8 * c)) & 0xFFu;
      const __half2 h1 = __float2half2_rn(-(1024.0f + (float)za)), h2 = __float2half2_rn(-(1024.0f + 16.0f * (float)za));
      const __half2 h3 = __float2half2_rn(-(1024.0f + (float)zb)), h4 = __float2half2_rn(-(1024.0f + 16.0f * (float)zb));
      ne_a = *reinterpret_cast<const uint32_t*>(&h1);
      no_a = *reinterpret_cast<const uint32_t*>(&h2);
      ne_b = *reinterpret_cast<const uint32_t*>(&h3);
      no_b = *reinterpret_cast<const uint32_t*>(&h4);
    }
    if (owner) {
      if (bvalid) {
        const uint4* src = reinterpret_cast<const uint4*>(sl + kSlotCode + kSlotScale + kSlotZp + oid * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 v = src[j * 8];
          bw[4 * j] = v.x; bw[4 * j + 1] = v.y; bw[4 * j + 2] = v.z; bw[4 * j + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) bw[j] = 0u;
      }
    }
    slot = slot + 1 == kRingB ? 0 : slot + 1;
    float s_a0, s_a1, s_b0, s_b1;
    if constexpr (BF16S) {
      s_a0 = __uint_as_float(swa << 16); s_a1 = __uint_as_float(swa & 0xFFFF0000u);
      s_b0 = __uint_as_float(swb << 16); s_b1 = __uint_as_float(swb & 0xFFFF0000u);
    } else {
      s_a0 = __half2float(__ushort_as_half((uint16_t)(swa & 0xFFFFu))); s_a1 = __half2float(__ushort_as_half((uint16_t)(swa >> 16)));
      s_b0 = __half2float(__ushort_as_half((uint16_t)(swb & 0xFFFFu))); s_b1 = __half2float(__ushort_as_half((uint16_t)(swb >> 16)));
    }
    // Two chains (even / odd steps), each with the raw and the bias MMA. The A
    // operands are the codes placed in the FP16 mantissa, cut per step: step
    // 2i uses nibbles 0,4 / 1,5 of word i, step 2i+1 nibbles 2,6 / 3,7.
    constexpr uint32_t kMagic = 0x64006400u;
    const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
    const uint32_t wb[4] = {cbv.x, cbv.y, cbv.z, cbv.w};
    float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t va8 = wa[i] >> 8, vb8 = wb[i] >> 8;
      mma16816(t0, lop3_and_or(wa[i], 0x000F000Fu, kMagic), lop3_and_or(wb[i], 0x000F000Fu, kMagic),
               lop3_and_or(wa[i], 0x00F000F0u, kMagic), lop3_and_or(wb[i], 0x00F000F0u, kMagic),
               bw[4 * i], bw[4 * i + 1]);
      mma16816(t1, lop3_and_or(va8, 0x000F000Fu, kMagic), lop3_and_or(vb8, 0x000F000Fu, kMagic),
               lop3_and_or(va8, 0x00F000F0u, kMagic), lop3_and_or(vb8, 0x00F000F0u, kMagic),
               bw[4 * i + 2], bw[4 * i + 3]);
      mma16816(t0, ne_a, ne_b, no_a, no_b, bw[4 * i], bw[4 * i + 1]);
      mma16816(t1, ne_a, ne_b, no_a, no_b, bw[4 * i + 2], bw[4 * i + 3]);
    }
    acc[0] = fmaf(s_a0, t0[0] + t1[0], acc[0]);
    acc[1] = fmaf(s_a1, t0[1] + t1[1], acc[1]);
    acc[2] = fmaf(s_b0, t0[2] + t1[2], acc[2]);
    acc[3] = fmaf(s_b1, t0[3] + t1[3], acc[3]);
    ++cic;
    if (cic < nq && f + 1 < total) continue;

    // ---- this warp's part of the unit is done
    const bool whole = first_cic == 0 && cic == nq;
    bool last = true;
    if (!whole) {
      // parts of this unit: the warps owning its first and last chunk, and those between
      const int64_t ux = (int64_t)item * nq;
      const int w0 = chunk_owner(ux, nw, cfull), w1 = chunk_owner(ux + nq - 1, nw, cfull);
      // partial slot 0: the piece's first unit; slot 1: its last unit
      float* part = ws.dsplit + ((size_t)wg * 2 + (item == item0 ? 0 : 1)) * 128;
#pragma unroll
      for (int r = 0; r < 4; ++r) part[r * 32 + lane] = acc[r];
      __syncwarp();
      int old = 0;
      if (lane == 0) {
        // release: the warp's partial tile is visible before the ticket moves;
        // acquire: the other parts' tiles are visible to the last arriver
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(ws.dticket + item) : "memory");
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      last = old == w1 - w0;
      if (last) {
        if (lane == 0) ws.dticket[item] = 0;    // free again for fc2 and the next call
        __syncwarp();
        // parts added in chunk order: warps w0 .. w1. Warp w0's piece may begin
        // before the unit (the unit is then its last, slot 1); every later
        // warp's piece begins inside it (slot 0).
        const int hs0 = cfull * w0 / nw < ux ? 1 : 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float v = 0.f;
          for (int wk = w0; wk <= w1; ++wk) {
            const int hs = wk == w0 ? hs0 : 0;
            const float pk = wk == wg ? acc[r] : __ldcg(ws.dsplit + ((size_t)wk * 2 + hs) * 128 + r * 32 + lane);
            v = wk == w0 ? pk : v + pk;
          }
          acc[r] = v;
        }
      }
    }
    if (last) {
      const int row0 = (item % rgroups) * kRowsPerGroup;
      // route sum over its four block columns: lanes c and c^1 hold two each
      float v_lo = acc[0] + acc[1];
      float v_hi = acc[2] + acc[3];
      v_lo += __shfl_xor_sync(0xffffffffu, v_lo, 1);
      v_hi += __shfl_xor_sync(0xffffffffu, v_hi, 1);
      const int n = c >> 1;                      // route within the pair of this lane's columns
      if constexpr (FC1) {
        const float up_lo = __shfl_down_sync(0xffffffffu, v_lo, 4);
        const float up_hi = __shfl_down_sync(0xffffffffu, v_hi, 4);
        if ((g & 1) == 0 && (c & 1) == 0 && n < cnt) {
          const int pos = pos0 + n;
          const float sigma = ws.tok_scale[n ? tok1 : tok0];
          const float inv = 1.0f / sigma;
          const int j_lo = row0 / 2 + g / 2, j_hi = j_lo + 4;
          const int ex = __ldg(ws.dtab + (item / rgroups) * kDtabInts);
          float2 b_lo = make_float2(0.0f, 0.0f), b_hi = b_lo;
          if (p.b1) {
            b_lo = fc1_bias_pair(p, ex, j_lo);
            b_hi = fc1_bias_pair(p, ex, j_hi);
          }
          const float hs = sigma * sigma * __int_as_float(__ldg(ws.dtab + (item / rgroups) * kDtabInts + 7));
          const float h_lo = silu(v_lo * inv + b_lo.x) * (up_lo * inv + b_lo.y) * hs;
          const float h_hi = silu(v_hi * inv + b_hi.x) * (up_hi * inv + b_hi.y) * hs;
          // fc2 reads these as activations: odd K positions carry 1/16
          ws.h16[(int64_t)pos * p.I + permuted_pos(j_lo, 8)] =
              __half_as_ushort(__float2half_rn((j_lo & 1) ? h_lo * 0.0625f : h_lo));
          ws.h16[(int64_t)pos * p.I + permuted_pos(j_hi, 8)] =
              __half_as_ushort(__float2half_rn((j_hi & 1) ? h_hi * 0.0625f : h_hi));
        }
      } else {
        if ((c & 1) == 0 && n < cnt) {
          const int rid = ws.sorted_route[pos0 + n];
          const float inv = 1.0f / ws.tok_scale[rid / p.k];
          const float hn = __int_as_float(__ldg(ws.dtab + (item / rgroups) * kDtabInts + 7));
          const float fct = inv * inv / hn * ws.topk_w[rid];
          ws.y[(int64_t)rid * p.H + row0 + g] = v_lo * fct;
          ws.y[(int64_t)rid * p.H + row0 + g + 8] = v_hi * fct;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r] = 0.f;
    if (cic == nq) { cic = 0; ++item; }
    first_cic = cic;
    fresh = true;
  }
  cp_async_wait<0>();
}

template <bool FC1, bool BF16S, bool HAS_ZP>
cudaError_t launch_int4_bs_t(DecodeArgs a, int64_t blocks, size_t smem, cudaStream_t s) {
  const cudaError_t err = ensure_smem_optin(decode_int4_bs_kernel<FC1, BF16S, HAS_ZP>, 75 * 1024);
  if (err != cudaSuccess) return err;
  return launch_pdl(decode_int4_bs_kernel<FC1, BF16S, HAS_ZP>, dim3((unsigned)blocks), dim3(32 * kWarps), smem, s, a);
}

int64_t decode_grid_blocks() { return (int64_t)sm_count() * kBlocksPerSmB; }

// ---------------------------------------------------------------------------
// INT4, block 32, K a multiple of 256: the same per-chunk arithmetic as above,
// with the operands brought in by the tensor-memory-access unit. Lane 0 of each
// warp issues, per 256-wide K chunk of a unit, four or five bulk tensor copies
// (codes as one [16 rows][128 B] box, the [16 rows][8] block scales, the
// chunk's activations of one or two tokens, the zero points when present) into
// the warp's ring slot, completing on the slot's mbarrier; the other lanes only
// wait on the barrier and read shared memory. Lanes that supply no activations
// read a zero area instead of branching. Work split, tickets and epilogues are
// those of the kernel above, with 256-wide chunks.
// ---------------------------------------------------------------------------
constexpr int kTWarps = 8;
constexpr int kTChunkK = 256;
constexpr int kTBlocksPerSm = 2;
constexpr int kTMinPiece = 2;                      // chunks per warp at least
constexpr int kTZero = 512;                        // zero bytes read by non-supplying lanes
constexpr uint64_t kTWaitNs = QMOE_WAIT_LIMIT_NS;
constexpr uint64_t kTDrainNs = 100000000ull;
constexpr int kErrDecodeTimeout = 2;

// Unit height: 16 rows (one MMA M-fragment) or 32 rows (two, sharing each
// chunk's activations: fewer instructions per weight byte, but longer units and
// a shallower ring in the same shared memory). Slot layout, every part 128-byte
// aligned: codes [ROWS][128 B] (sub-chunk s at byte 64 s), scales [ROWS][8],
// zero points [ROWS][16], activations of the pair's two tokens [256] FP16 each.
template <int ROWS>
struct TCfg {
  static constexpr int kRows = ROWS;
  static constexpr int kHalves = ROWS / 16;
  static constexpr int kRing = ROWS == 32 ? 2 : 3;   // chunks per warp: kRing - 1 in flight, one in use
  static constexpr int kCode = 0;
  static constexpr int kScale = ROWS * 128;
  static constexpr int kZp = kScale + ROWS * 16;
  static constexpr int kAct0 = kZp + ROWS * 16;
  static constexpr int kAct1 = kAct0 + 512;
  static constexpr int kSlot = kAct1 + 512;
  static constexpr int kPart = kHalves * 4 * 32;      // FP32 partial tile of one unit
  static constexpr size_t kSmem = (size_t)kTWarps * kRing * kSlot + kTZero + kTWarps * kRing * 8 + 128;
};
constexpr int kTPartMax = TCfg<32>::kPart;

struct TmaDecodeArgs {
  int N, K;
  Problem p;
  Workspace ws;
};

template <int ROWS, bool FC1, bool BF16S, bool HAS_ZP>
__global__ void __launch_bounds__(32 * kTWarps, kTBlocksPerSm) decode_int4_tma_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap ts,
    const __grid_constant__ CUtensorMap tz, const __grid_constant__ CUtensorMap ta, TmaDecodeArgs a) {
  using C = TCfg<ROWS>;
  // fc1 needs the routing kernel's results at once. fc2 reads only the routing
  // results (complete: fc1 let fc2 be scheduled only after waiting for routing)
  // and its own weights before it waits for fc1, so its first weight copies
  // overlap the end of fc1.
  if constexpr (FC1) {
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_trigger();
  }
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  const int K = a.K, N = a.N;
  const int nq = K / kTChunkK;                   // chunks per unit
  const int rgroups = N / C::kRows;
  const int cfull = ws.counters[3] * rgroups * nq;   // < 2^31: <= 256 entries x 512 groups x 32 chunks

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int gw = gridDim.x * kTWarps;
  const int wg = blockIdx.x * kTWarps + warp;
  // equal pieces of L chunks (the last one shorter, none empty)
  int L = (cfull + gw - 1) / gw;
  if (L < kTMinPiece) L = kTMinPiece;
  const int nw = (cfull + L - 1) / L;
  const int x_begin = wg < nw ? wg * L : 0;
  const int total = wg < nw ? min(x_begin + L, cfull) - x_begin : 0;
  const bool owner = (g & 3) == c;               // supplies activations for column g
  const int on = g >> 2;                         // owner lane's route within the pair
  const int n = c >> 1;                          // route within the pair of this lane's D columns

  extern __shared__ __align__(16) uint8_t smem[];
  // bulk tensor copies land on 128-byte boundaries
  uint8_t* base = smem + ((128u - (smem_u32(smem) & 127u)) & 127u);
  const uint32_t ring_s = smem_u32(base) + warp * (C::kRing * C::kSlot);
  const uint32_t zero_s = smem_u32(base) + kTWarps * C::kRing * C::kSlot;
  const uint32_t bar_s = zero_s + kTZero + warp * (C::kRing * 8);
  if (threadIdx.x < kTZero / 4) reinterpret_cast<uint32_t*>(base + kTWarps * C::kRing * C::kSlot)[threadIdx.x] = 0u;
  if (lane == 0)
    for (int s = 0; s < C::kRing; ++s) mbar_init(bar_s + 8 * s, 1);
  mbar_init_fence();
  __syncthreads();
  if (total == 0) {
    if constexpr (!FC1) pdl_wait();
    return;
  }

  // unit = (decode-table entry ei, 32-row group rg); walked without divisions
  const int item0 = x_begin / nq;
  const int cic0 = x_begin - item0 * nq;
  const int ei0 = item0 / rgroups, rg0 = item0 - ei0 * rgroups;

  // ---- issue side: lane 0 copies chunk f of the piece into slot f % C::kRing:
  // the weights (codes, scales, zero points; announced without arriving) and the
  // activations of the entry's tokens (announced with the arrival)
  int p_ei = ei0, p_rg = rg0, p_cic = cic0, p_row = 0, p_t0 = 0, p_t1 = 0, p_cnt = 0;
  bool p_new = true;
  uint32_t p_slot_s = ring_s, p_bar = bar_s;
  auto issue_act = [&](uint32_t slot_s, uint32_t bar, int kx, int t0, int t1, int cnt) {
    if (lane == 0) {
      mbar_expect_tx(bar, cnt > 1 ? 1024 : 512);
      tma_load_2d(slot_s + C::kAct0, &ta, bar, kx, t0);
      if (cnt > 1) tma_load_2d(slot_s + C::kAct1, &ta, bar, kx, t1);
    }
  };
  // deferred activation copies of the first slots (fc2: issued after the wait)
  uint32_t q_slot[C::kRing - 1], q_bar[C::kRing - 1];
  int q_kx[C::kRing - 1], q_t0[C::kRing - 1], q_t1[C::kRing - 1], q_cnt[C::kRing - 1];
  auto issue = [&](bool with_act, int q) {
    if (p_new) {
      p_new = false;
      const int4 d0 = __ldg(reinterpret_cast<const int4*>(ws.dtab + p_ei * kDtabInts));
      const int4 d1 = __ldg(reinterpret_cast<const int4*>(ws.dtab + p_ei * kDtabInts + 4));
      p_row = d0.x * N + p_rg * C::kRows;
      p_cnt = d0.z;
      p_t0 = FC1 ? d1.x : d0.y;
      p_t1 = FC1 ? d1.y : d0.y + 1;
    }
    const int kx = p_cic * kTChunkK;
    if (lane == 0) {
      mbar_expect_tx_only(p_bar, ROWS * 128 + ROWS * 16 + (HAS_ZP ? ROWS * 16 : 0));
      tma_load_2d(p_slot_s + C::kCode, &tq, p_bar, kx / 2, p_row);
      tma_load_2d(p_slot_s + C::kScale, &ts, p_bar, kx / 32, p_row);
      if constexpr (HAS_ZP) tma_load_2d(p_slot_s + C::kZp, &tz, p_bar, (kx / 32) & ~15, p_row);
    }
    if (with_act) {
      issue_act(p_slot_s, p_bar, kx, p_t0, p_t1, p_cnt);
    } else {
      q_slot[q] = p_slot_s; q_bar[q] = p_bar; q_kx[q] = kx; q_t0[q] = p_t0; q_t1[q] = p_t1; q_cnt[q] = p_cnt;
    }
    if (p_bar == bar_s + 8 * (C::kRing - 1)) { p_bar = bar_s; p_slot_s = ring_s; }
    else { p_bar += 8; p_slot_s += C::kSlot; }
    if (++p_cic == nq) {
      p_cic = 0;
      p_new = true;
      if (++p_rg == rgroups) { p_rg = 0; ++p_ei; }
    }
  };
  const int pre = total < C::kRing - 1 ? total : C::kRing - 1;
#pragma unroll
  for (int u = 0; u < C::kRing - 1; ++u)
    if (u < pre) issue(FC1, u);
  if constexpr (!FC1) {
    pdl_wait();                                  // h16 (fc1's output) is complete from here on
#pragma unroll
    for (int u = 0; u < C::kRing - 1; ++u)
      if (u < pre) issue_act(q_slot[u], q_bar[u], q_kx[u], q_t0[u], q_t1[u], q_cnt[u]);
  }

  const __half2 ne_d = __float2half2_rn(-(1024.0f + 8.0f)), no_d = __float2half2_rn(-(1024.0f + 128.0f));
  const uint32_t ne_def = *reinterpret_cast<const uint32_t*>(&ne_d);
  const uint32_t no_def = *reinterpret_cast<const uint32_t*>(&no_d);
  // per-lane shared-memory offsets within a slot (the rest are immediates)
  const uint32_t code_off = g * 128 + c * 16;   // row g of the [16][128 B] code tile
  const uint32_t scale_off = C::kScale + g * 16 + 4 * (c & 1);
  // activation words: owners read their token's tile, the other lanes the zero area
  const uint32_t act_base = owner ? ring_s + (on ? C::kAct1 : C::kAct0) + 64 * c : zero_s;
  const uint32_t act_slot_stride = owner ? C::kSlot : 0;

  // ---- compute side
  int ei = ei0, rg = rg0, cic = cic0, first_cic = cic0;
  bool first_unit = true, fresh = true;
  int cnt = 0, pos0 = 0, e_rid = 0;
  float e_scale = 1.0f, e_w = 0.0f;              // epilogue operands of route n, loaded early
  float e_hn = 1.0f;                             // the expert's SwiGLU normalisation (decode table)
  float acc[C::kHalves][4];                    // [row half][D fragment]
#pragma unroll
  for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[rh][r] = 0.f;
  int slot = 0;
  uint32_t phase = 0;
  for (int f = 0; f < total; ++f) {
    __syncwarp();                                // every lane is done with the slot refilled next
    if (f + C::kRing - 1 < total) issue(true, 0);
    if (fresh) {
      fresh = false;
      const int4 d0 = __ldg(reinterpret_cast<const int4*>(ws.dtab + ei * kDtabInts));
      const int4 d1 = __ldg(reinterpret_cast<const int4*>(ws.dtab + ei * kDtabInts + 4));
      pos0 = d0.y;
      cnt = d0.z;
      e_hn = __int_as_float(d1.w);
      if (n < cnt) {
        if constexpr (FC1) {
          e_scale = __ldg(ws.tok_scale + (n ? d1.y : d1.x));
        } else {
          e_rid = __ldg(ws.sorted_route + pos0 + n);
          e_scale = __ldg(ws.tok_scale + e_rid / p.k);
          e_w = __ldg(ws.topk_w + e_rid);
        }
      }
    }
    const uint32_t bar = bar_s + 8 * slot;
    if (!mbar_wait_for(bar, phase, kTWaitNs)) {
      // record the failure, let this warp's copies in flight land, and stop
      if (lane == 0) atomicExch(ws.counters + 2, kErrDecodeTimeout);
      int s2 = slot;
      uint32_t ph2 = phase;
      const int inflight = total - f < C::kRing ? total - f : C::kRing;   // chunks f .. f + C::kRing - 1
      for (int u = 0; u < inflight; ++u) {
        mbar_wait_for(bar_s + 8 * s2, ph2, kTDrainNs);
        if (++s2 == C::kRing) { s2 = 0; ph2 ^= 1u; }
      }
      return;
    }
    const uint32_t sb = ring_s + slot * C::kSlot;
    const uint32_t ab = act_base + slot * act_slot_stride;
    // the activations (B fragments) of both sub-chunks serve both 16-row halves
    uint32_t bw[2][16];
#define QMOE_LDS_ACT(SUB, J, OFF)                                                                  \
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+" #OFF "];\n"                                 \
               : "=r"(bw[SUB][4 * J]), "=r"(bw[SUB][4 * J + 1]), "=r"(bw[SUB][4 * J + 2]),         \
                 "=r"(bw[SUB][4 * J + 3])                                                          \
               : "r"(ab))
    QMOE_LDS_ACT(0, 0, 0);
    QMOE_LDS_ACT(0, 1, 16);
    QMOE_LDS_ACT(0, 2, 32);
    QMOE_LDS_ACT(0, 3, 48);
    QMOE_LDS_ACT(1, 0, 256);
    QMOE_LDS_ACT(1, 1, 272);
    QMOE_LDS_ACT(1, 2, 288);
    QMOE_LDS_ACT(1, 3, 304);
#undef QMOE_LDS_ACT
    // With the implicit zero point every weight row has the same bias operand, so
    // the bias MMAs are computed once per chunk and start each row half's sums.
    float tb[2][2][4];
#pragma unroll
    for (int sub = 0; sub < 2; ++sub)
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) tb[sub][q][e] = 0.f;
    if constexpr (!HAS_ZP) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          mma16816(tb[sub][0], ne_def, ne_def, no_def, no_def, bw[sub][4 * i], bw[sub][4 * i + 1]);
          mma16816(tb[sub][1], ne_def, ne_def, no_def, no_def, bw[sub][4 * i + 2], bw[sub][4 * i + 3]);
        }
    }
#pragma unroll
    for (int rh = 0; rh < C::kHalves; ++rh) {
      const uint32_t cb_ = sb + code_off + rh * 2048, sr = sb + scale_off + rh * 256;   // rows 16 rh ..
      uint4 cw[2][2];
      uint32_t sw[2][2];
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(cw[0][0].x), "=r"(cw[0][0].y), "=r"(cw[0][0].z), "=r"(cw[0][0].w) : "r"(cb_));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+1024];\n"
                   : "=r"(cw[0][1].x), "=r"(cw[0][1].y), "=r"(cw[0][1].z), "=r"(cw[0][1].w) : "r"(cb_));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+64];\n"
                   : "=r"(cw[1][0].x), "=r"(cw[1][0].y), "=r"(cw[1][0].z), "=r"(cw[1][0].w) : "r"(cb_));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+1088];\n"
                   : "=r"(cw[1][1].x), "=r"(cw[1][1].y), "=r"(cw[1][1].z), "=r"(cw[1][1].w) : "r"(cb_));
      asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(sw[0][0]) : "r"(sr));
      asm volatile("ld.shared.u32 %0, [%1+128];\n" : "=r"(sw[0][1]) : "r"(sr));
      asm volatile("ld.shared.u32 %0, [%1+8];\n" : "=r"(sw[1][0]) : "r"(sr));
      asm volatile("ld.shared.u32 %0, [%1+136];\n" : "=r"(sw[1][1]) : "r"(sr));
      uint32_t ne_a[2], ne_b[2], no_a[2], no_b[2];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        ne_a[sub] = ne_def; ne_b[sub] = ne_def; no_a[sub] = no_def; no_b[sub] = no_def;
        if constexpr (HAS_ZP) {
          uint32_t zwa, zwb;
          const uint32_t zrow = sb + C::kZp + (rh * 16 + g) * 16 + (cic & 1) * 8 + 4 * sub;
          asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(zwa) : "r"(zrow));
          asm volatile("ld.shared.u32 %0, [%1+128];\n" : "=r"(zwb) : "r"(zrow));
          const uint32_t za = (zwa >> (8 * c)) & 0xFFu, zb = (zwb >> (8 * c)) & 0xFFu;
          const __half2 h1 = __float2half2_rn(-(1024.0f + (float)za)), h2 = __float2half2_rn(-(1024.0f + 16.0f * (float)za));
          const __half2 h3 = __float2half2_rn(-(1024.0f + (float)zb)), h4 = __float2half2_rn(-(1024.0f + 16.0f * (float)zb));
          ne_a[sub] = *reinterpret_cast<const uint32_t*>(&h1);
          no_a[sub] = *reinterpret_cast<const uint32_t*>(&h2);
          ne_b[sub] = *reinterpret_cast<const uint32_t*>(&h3);
          no_b[sub] = *reinterpret_cast<const uint32_t*>(&h4);
        }
      }
      constexpr uint32_t kMagic = 0x64006400u;
      float t[2][2][4];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) t[sub][q][e] = tb[sub][q][e];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const uint32_t wa = (&cw[sub][0].x)[i], wb = (&cw[sub][1].x)[i];
          const uint32_t va8 = wa >> 8, vb8 = wb >> 8;
          mma16816(t[sub][0], lop3_and_or(wa, 0x000F000Fu, kMagic), lop3_and_or(wb, 0x000F000Fu, kMagic),
                   lop3_and_or(wa, 0x00F000F0u, kMagic), lop3_and_or(wb, 0x00F000F0u, kMagic),
                   bw[sub][4 * i], bw[sub][4 * i + 1]);
          mma16816(t[sub][1], lop3_and_or(va8, 0x000F000Fu, kMagic), lop3_and_or(vb8, 0x000F000Fu, kMagic),
                   lop3_and_or(va8, 0x00F000F0u, kMagic), lop3_and_or(vb8, 0x00F000F0u, kMagic),
                   bw[sub][4 * i + 2], bw[sub][4 * i + 3]);
        }
        if constexpr (HAS_ZP) {
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            mma16816(t[sub][0], ne_a[sub], ne_b[sub], no_a[sub], no_b[sub], bw[sub][4 * i], bw[sub][4 * i + 1]);
            mma16816(t[sub][1], ne_a[sub], ne_b[sub], no_a[sub], no_b[sub], bw[sub][4 * i + 2], bw[sub][4 * i + 3]);
          }
        }
      }
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        float s_a0, s_a1, s_b0, s_b1;
        const uint32_t swa = sw[sub][0], swb = sw[sub][1];
        if constexpr (BF16S) {
          s_a0 = __uint_as_float(swa << 16); s_a1 = __uint_as_float(swa & 0xFFFF0000u);
          s_b0 = __uint_as_float(swb << 16); s_b1 = __uint_as_float(swb & 0xFFFF0000u);
        } else {
          s_a0 = __half2float(__ushort_as_half((uint16_t)(swa & 0xFFFFu))); s_a1 = __half2float(__ushort_as_half((uint16_t)(swa >> 16)));
          s_b0 = __half2float(__ushort_as_half((uint16_t)(swb & 0xFFFFu))); s_b1 = __half2float(__ushort_as_half((uint16_t)(swb >> 16)));
        }
        acc[rh][0] = fmaf(s_a0, t[sub][0][0] + t[sub][1][0], acc[rh][0]);
        acc[rh][1] = fmaf(s_a1, t[sub][0][1] + t[sub][1][1], acc[rh][1]);
        acc[rh][2] = fmaf(s_b0, t[sub][0][2] + t[sub][1][2], acc[rh][2]);
        acc[rh][3] = fmaf(s_b1, t[sub][0][3] + t[sub][1][3], acc[rh][3]);
      }
    }
    if (++slot == C::kRing) { slot = 0; phase ^= 1u; }
    if (++cic < nq && f + 1 < total) continue;

    // ---- this warp's part of the unit is done
    const bool whole = first_cic == 0 && cic == nq;
    bool last = true;
    if (!whole) {
      // parts of this unit: the warps owning its first and last chunk, and those between
      const int item = ei * rgroups + rg;
      const int ux = item * nq;
      const int w0 = ux / L, w1 = (ux + nq - 1) / L;
      // partial slot 0: the piece's first unit; slot 1: its last unit
      float* part = ws.dsplit + ((size_t)wg * 2 + (first_unit ? 0 : 1)) * C::kPart;
#pragma unroll
      for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
        for (int r = 0; r < 4; ++r) part[(rh * 4 + r) * 32 + lane] = acc[rh][r];
      __syncwarp();
      int old = 0;
      if (lane == 0) {
        // release: the warp's partial tile is visible before the ticket moves;
        // acquire: the other parts' tiles are visible to the last arriver
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(ws.dticket + item) : "memory");
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      last = old == w1 - w0;
      if (last) {
        if (lane == 0) ws.dticket[item] = 0;    // free again for fc2 and the next call
        __syncwarp();
        // parts added in chunk order: warps w0 .. w1. Warp w0's piece may begin
        // before the unit (the unit is then its last, slot 1); every later
        // warp's piece begins inside it (slot 0).
        const int hs0 = w0 * L < ux ? 1 : 0;
#pragma unroll
        for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float v = 0.f;
            for (int wk = w0; wk <= w1; ++wk) {
              const int hs = wk == w0 ? hs0 : 0;
              const float pk = wk == wg ? acc[rh][r]
                                        : __ldcg(ws.dsplit + ((size_t)wk * 2 + hs) * C::kPart + (rh * 4 + r) * 32 + lane);
              v = wk == w0 ? pk : v + pk;
            }
            acc[rh][r] = v;
          }
      }
    }
    if (last) {
#pragma unroll
      for (int rh = 0; rh < C::kHalves; ++rh) {
      const int row0 = rg * C::kRows + rh * kRowsPerGroup;
      float v_lo = acc[rh][0] + acc[rh][1];
      float v_hi = acc[rh][2] + acc[rh][3];
      v_lo += __shfl_xor_sync(0xffffffffu, v_lo, 1);
      v_hi += __shfl_xor_sync(0xffffffffu, v_hi, 1);
      if constexpr (FC1) {
        const float up_lo = __shfl_down_sync(0xffffffffu, v_lo, 4);
        const float up_hi = __shfl_down_sync(0xffffffffu, v_hi, 4);
        if ((g & 1) == 0 && (c & 1) == 0 && n < cnt) {
          const int pos = pos0 + n;
          const float sigma = e_scale;
          const float inv = 1.0f / sigma;
          const int j_lo = row0 / 2 + g / 2, j_hi = j_lo + 4;
          const int ex = __ldg(ws.dtab + ei * kDtabInts);
          float2 b_lo = make_float2(0.0f, 0.0f), b_hi = b_lo;
          if (p.b1) {
            b_lo = fc1_bias_pair(p, ex, j_lo);
            b_hi = fc1_bias_pair(p, ex, j_hi);
          }
          const float hs = sigma * sigma * e_hn;
          const float h_lo = silu(v_lo * inv + b_lo.x) * (up_lo * inv + b_lo.y) * hs;
          const float h_hi = silu(v_hi * inv + b_hi.x) * (up_hi * inv + b_hi.y) * hs;
          // fc2 reads these as activations: odd K positions carry 1/16
          ws.h16[(int64_t)pos * p.I + permuted_pos(j_lo, 8)] =
              __half_as_ushort(__float2half_rn((j_lo & 1) ? h_lo * 0.0625f : h_lo));
          ws.h16[(int64_t)pos * p.I + permuted_pos(j_hi, 8)] =
              __half_as_ushort(__float2half_rn((j_hi & 1) ? h_hi * 0.0625f : h_hi));
        }
      } else {
        if ((c & 1) == 0 && n < cnt) {
          const float inv = 1.0f / e_scale;
          const float fct = inv * inv / e_hn * e_w;
          ws.y[(int64_t)e_rid * p.H + row0 + g] = v_lo * fct;
          ws.y[(int64_t)e_rid * p.H + row0 + g + 8] = v_hi * fct;
        }
      }
      }
    }
#pragma unroll
    for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[rh][r] = 0.f;
    if (cic == nq) {
      cic = 0;
      if (++rg == rgroups) { rg = 0; ++ei; }
    }
    first_cic = cic;
    first_unit = false;
    fresh = true;
  }
}

// ---------------------------------------------------------------------------
// INT3 and INT2 (implicit zero points 4 and 2), blocks of 32, 64 or 128, K a
// multiple of 256: the tensor-copy kernel's walk, tickets and epilogues with
// 3- or 2-bit codes. A chunk's codes are one [rows][32 * BITS bytes] box; lane
// c takes its 32 codes of a 128-wide half as 4 * BITS bytes (INT3: byte permutes
// put two 8-code groups in the two 16-bit halves), and one shift and one
// AND/OR per pair give 1024 + code in FP16, in the same 16-group K permutation
// as the activations. One bias MMA per K step (operand -(1024 + zp)) is shared
// by all row halves. The block
// scales come by one 16-, 8- or 4-byte load per lane and row, stored into the
// slot one chunk later (scale rows need not be a multiple of 16 bytes, as a
// tensor copy would require); each D column takes the scale of the block its
// owner lane's codes fall in.
// ---------------------------------------------------------------------------
template <int BITS, int ROWS>
struct T23Cfg {
  static constexpr int kRows = ROWS;
  static constexpr int kHalves = ROWS / 16;
  static constexpr int kRing = 3;                     // chunks per warp: two in flight, one in use
  static constexpr int kCodeRow = 32 * BITS;          // code bytes of a row in a 256-wide chunk
  static constexpr int kCode = 0;                     // [ROWS][kCodeRow]
  static constexpr int kScale = ROWS * kCodeRow;      // [ROWS][8] 16-bit scales (the first 8, 4 or 2 used)
  static constexpr int kAct0 = kScale + ROWS * 16;
  static constexpr int kAct1 = kAct0 + 512;
  static constexpr int kSlot = kAct1 + 512;
  static constexpr int kPart = kHalves * 4 * 32;
  static constexpr size_t kSmem = (size_t)kTWarps * kRing * kSlot + kTZero + kTWarps * kRing * 8 + 128;
  static_assert(kScale % 128 == 0 && kAct0 % 128 == 0 && kSlot % 128 == 0, "copies land on 128-byte boundaries");
};

struct Tma23Args {
  int N, K;
  Problem p;
  Workspace ws;
  const uint16_t* s;       // [E][N][K/block] block scales in dtype
  int lb;                  // log2(block)
};

template <int BITS, int ROWS, bool FC1, bool BF16S>
__global__ void __launch_bounds__(32 * kTWarps, kTBlocksPerSm) decode_int23_tma_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap ta, Tma23Args a) {
  static_assert(BITS == 2 || BITS == 3, "3- or 2-bit codes");
  using C = T23Cfg<BITS, ROWS>;
  // fc1 needs the routing kernel's results at once. fc2 reads only the routing
  // results (complete: fc1 let fc2 be scheduled only after waiting for routing)
  // and its own weights before it waits for fc1, so its first weight copies
  // overlap the end of fc1.
  if constexpr (FC1) {
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_trigger();
  }
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  const int K = a.K, N = a.N;
  const int nq = K / kTChunkK;                   // chunks per unit
  const int rgroups = N / C::kRows;
  const int cfull = ws.counters[3] * rgroups * nq;   // < 2^31: <= 256 entries x 512 groups x 32 chunks

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int gw = gridDim.x * kTWarps;
  const int wg = blockIdx.x * kTWarps + warp;
  // equal pieces of L chunks (the last one shorter, none empty)
  int L = (cfull + gw - 1) / gw;
  if (L < kTMinPiece) L = kTMinPiece;
  const int nw = (cfull + L - 1) / L;
  const int x_begin = wg < nw ? wg * L : 0;
  const int total = wg < nw ? min(x_begin + L, cfull) - x_begin : 0;
  const bool owner = (g & 3) == c;               // supplies activations for column g
  const int on = g >> 2;                         // owner lane's route within the pair
  const int n = c >> 1;                          // route within the pair of this lane's D columns

  extern __shared__ __align__(16) uint8_t smem[];
  // bulk tensor copies land on 128-byte boundaries
  uint8_t* base = smem + ((128u - (smem_u32(smem) & 127u)) & 127u);
  const uint32_t ring_s = smem_u32(base) + warp * (C::kRing * C::kSlot);
  const uint32_t zero_s = smem_u32(base) + kTWarps * C::kRing * C::kSlot;
  const uint32_t bar_s = zero_s + kTZero + warp * (C::kRing * 8);
  if (threadIdx.x < kTZero / 4) reinterpret_cast<uint32_t*>(base + kTWarps * C::kRing * C::kSlot)[threadIdx.x] = 0u;
  if (lane == 0)
    for (int s = 0; s < C::kRing; ++s) mbar_init(bar_s + 8 * s, 1);
  mbar_init_fence();
  __syncthreads();
  if (total == 0) {
    if constexpr (!FC1) pdl_wait();
    return;
  }

  // unit = (decode-table entry ei, 32-row group rg); walked without divisions
  const int item0 = x_begin / nq;
  const int cic0 = x_begin - item0 * nq;
  const int ei0 = item0 / rgroups, rg0 = item0 - ei0 * rgroups;

  // ---- issue side: lane 0 copies chunk f of the piece into slot f % C::kRing:
  // the weights (codes, scales, zero points; announced without arriving) and the
  // activations of the entry's tokens (announced with the arrival)
  int p_ei = ei0, p_rg = rg0, p_cic = cic0, p_row = 0, p_t0 = 0, p_t1 = 0, p_cnt = 0;
  bool p_new = true;
  uint32_t p_slot_s = ring_s, p_bar = bar_s;
  // block scales: lane L < ROWS loads row L's scales of the chunk (16, 8 or 4
  // bytes for blocks of 32, 64 or 128) when the chunk is issued and stores them
  // into the slot one chunk later, so that the load's latency is hidden
  const int lb = a.lb;
  const int nblk = K >> lb;
  uint4 s_pend = make_uint4(0u, 0u, 0u, 0u);
  uint32_t s_pend_dst = 0;
  bool s_have = false;
  auto scale_store = [&]() {
    if (s_have && lane < ROWS) {
      if (lb == 5)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(s_pend_dst), "r"(s_pend.x), "r"(s_pend.y),
                     "r"(s_pend.z), "r"(s_pend.w) : "memory");
      else if (lb == 6)
        asm volatile("st.shared.v2.u32 [%0], {%1,%2};\n" ::"r"(s_pend_dst), "r"(s_pend.x), "r"(s_pend.y) : "memory");
      else
        asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(s_pend_dst), "r"(s_pend.x) : "memory");
    }
    s_have = false;
  };
  auto issue_act = [&](uint32_t slot_s, uint32_t bar, int kx, int t0, int t1, int cnt) {
    if (lane == 0) {
      mbar_expect_tx(bar, cnt > 1 ? 1024 : 512);
      tma_load_2d(slot_s + C::kAct0, &ta, bar, kx, t0);
      if (cnt > 1) tma_load_2d(slot_s + C::kAct1, &ta, bar, kx, t1);
    }
  };
  // deferred activation copies of the first slots (fc2: issued after the wait)
  uint32_t q_slot[C::kRing - 1], q_bar[C::kRing - 1];
  int q_kx[C::kRing - 1], q_t0[C::kRing - 1], q_t1[C::kRing - 1], q_cnt[C::kRing - 1];
  auto issue = [&](bool with_act, int q) {
    if (p_new) {
      p_new = false;
      const int4 d0 = __ldg(reinterpret_cast<const int4*>(ws.dtab + p_ei * kDtabInts));
      const int4 d1 = __ldg(reinterpret_cast<const int4*>(ws.dtab + p_ei * kDtabInts + 4));
      p_row = d0.x * N + p_rg * C::kRows;
      p_cnt = d0.z;
      p_t0 = FC1 ? d1.x : d0.y;
      p_t1 = FC1 ? d1.y : d0.y + 1;
    }
    const int kx = p_cic * kTChunkK;
    if (lane == 0) {
      mbar_expect_tx_only(p_bar, ROWS * C::kCodeRow);
      tma_load_2d(p_slot_s + C::kCode, &tq, p_bar, kx / 8 * BITS, p_row);
    }
    // the previous chunk's scales go to its slot; this chunk's are loaded
    scale_store();
    if (lane < ROWS) {
      const uint16_t* src = a.s + (int64_t)(p_row + lane) * nblk + (kx >> lb);
      if (lb == 5) s_pend = __ldg(reinterpret_cast<const uint4*>(src));
      else if (lb == 6) { const uint2 v = __ldg(reinterpret_cast<const uint2*>(src)); s_pend.x = v.x; s_pend.y = v.y; }
      else s_pend.x = __ldg(reinterpret_cast<const uint32_t*>(src));
    }
    s_pend_dst = p_slot_s + C::kScale + lane * 16;
    s_have = true;
    if (with_act) {
      issue_act(p_slot_s, p_bar, kx, p_t0, p_t1, p_cnt);
    } else {
      q_slot[q] = p_slot_s; q_bar[q] = p_bar; q_kx[q] = kx; q_t0[q] = p_t0; q_t1[q] = p_t1; q_cnt[q] = p_cnt;
    }
    if (p_bar == bar_s + 8 * (C::kRing - 1)) { p_bar = bar_s; p_slot_s = ring_s; }
    else { p_bar += 8; p_slot_s += C::kSlot; }
    if (++p_cic == nq) {
      p_cic = 0;
      p_new = true;
      if (++p_rg == rgroups) { p_rg = 0; ++p_ei; }
    }
  };
  const int pre = total < C::kRing - 1 ? total : C::kRing - 1;
#pragma unroll
  for (int u = 0; u < C::kRing - 1; ++u)
    if (u < pre) issue(FC1, u);
  if constexpr (!FC1) {
    pdl_wait();                                  // h16 (fc1's output) is complete from here on
#pragma unroll
    for (int u = 0; u < C::kRing - 1; ++u)
      if (u < pre) issue_act(q_slot[u], q_bar[u], q_kx[u], q_t0[u], q_t1[u], q_cnt[u]);
  }

  // the implicit zero point 2^(BITS-1) of every code: -(1024 + zp) in every FP16 operand
  const __half2 nb_d = __float2half2_rn(-(1024.0f + (float)(1 << (BITS - 1))));
  const uint32_t nb_def = *reinterpret_cast<const uint32_t*>(&nb_d);
  // per-lane shared-memory offsets within a slot
  const uint32_t code_off = g * C::kCodeRow + c * (4 * BITS);   // row g of the code tile, lane c's 32 codes
  // the blocks of this lane's two D columns (owner lanes 2c & 3 and (2c + 1) & 3) in each 128-wide half
  // of the chunk, as byte offsets into a row's scales
  uint32_t blk_off[2][2];
#pragma unroll
  for (int sub = 0; sub < 2; ++sub) {
    blk_off[sub][0] = 2u * (uint32_t)((sub * 128 + ((2 * c) & 3) * 32) >> lb);
    blk_off[sub][1] = 2u * (uint32_t)((sub * 128 + ((2 * c + 1) & 3) * 32) >> lb);
  }
  // activation words: owners read their token's tile, the other lanes the zero area
  const uint32_t act_base = owner ? ring_s + (on ? C::kAct1 : C::kAct0) + 64 * c : zero_s;
  const uint32_t act_slot_stride = owner ? C::kSlot : 0;

  // ---- compute side
  int ei = ei0, rg = rg0, cic = cic0, first_cic = cic0;
  bool first_unit = true, fresh = true;
  int cnt = 0, pos0 = 0, e_rid = 0;
  float e_scale = 1.0f, e_w = 0.0f;              // epilogue operands of route n, loaded early
  float e_hn = 1.0f;                             // the expert's SwiGLU normalisation (decode table)
  float acc[C::kHalves][4];                    // [row half][D fragment]
#pragma unroll
  for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[rh][r] = 0.f;
  int slot = 0;
  uint32_t phase = 0;
  for (int f = 0; f < total; ++f) {
    __syncwarp();                                // every lane is done with the slot refilled next
    if (f + C::kRing - 1 < total) issue(true, 0);
    else scale_store();
    __syncwarp();                                // chunk f's scales are in its slot
    if (fresh) {
      fresh = false;
      const int4 d0 = __ldg(reinterpret_cast<const int4*>(ws.dtab + ei * kDtabInts));
      const int4 d1 = __ldg(reinterpret_cast<const int4*>(ws.dtab + ei * kDtabInts + 4));
      pos0 = d0.y;
      cnt = d0.z;
      e_hn = __int_as_float(d1.w);
      if (n < cnt) {
        if constexpr (FC1) {
          e_scale = __ldg(ws.tok_scale + (n ? d1.y : d1.x));
        } else {
          e_rid = __ldg(ws.sorted_route + pos0 + n);
          e_scale = __ldg(ws.tok_scale + e_rid / p.k);
          e_w = __ldg(ws.topk_w + e_rid);
        }
      }
    }
    const uint32_t bar = bar_s + 8 * slot;
    if (!mbar_wait_for(bar, phase, kTWaitNs)) {
      // record the failure, let this warp's copies in flight land, and stop
      if (lane == 0) atomicExch(ws.counters + 2, kErrDecodeTimeout);
      int s2 = slot;
      uint32_t ph2 = phase;
      const int inflight = total - f < C::kRing ? total - f : C::kRing;   // chunks f .. f + C::kRing - 1
      for (int u = 0; u < inflight; ++u) {
        mbar_wait_for(bar_s + 8 * s2, ph2, kTDrainNs);
        if (++s2 == C::kRing) { s2 = 0; ph2 ^= 1u; }
      }
      return;
    }
    const uint32_t sb = ring_s + slot * C::kSlot;
    const uint32_t ab = act_base + slot * act_slot_stride;
    // the activations (B fragments) of both sub-chunks serve both 16-row halves
    uint32_t bw[2][16];
#define QMOE_LDS_ACT(SUB, J, OFF)                                                                  \
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+" #OFF "];\n"                                 \
               : "=r"(bw[SUB][4 * J]), "=r"(bw[SUB][4 * J + 1]), "=r"(bw[SUB][4 * J + 2]),         \
                 "=r"(bw[SUB][4 * J + 3])                                                          \
               : "r"(ab))
    QMOE_LDS_ACT(0, 0, 0);
    QMOE_LDS_ACT(0, 1, 16);
    QMOE_LDS_ACT(0, 2, 32);
    QMOE_LDS_ACT(0, 3, 48);
    QMOE_LDS_ACT(1, 0, 256);
    QMOE_LDS_ACT(1, 1, 272);
    QMOE_LDS_ACT(1, 2, 288);
    QMOE_LDS_ACT(1, 3, 304);
#undef QMOE_LDS_ACT
    // Every weight row has the same bias operand (the implicit zero point), so
    // the bias MMAs are computed once per chunk and start each row half's sums:
    // stream q takes the K steps j with j % 2 == q.
    float tb[2][2][4];
#pragma unroll
    for (int sub = 0; sub < 2; ++sub)
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) tb[sub][q][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
        mma16816(tb[sub][j & 1], nb_def, nb_def, nb_def, nb_def, bw[sub][2 * j], bw[sub][2 * j + 1]);
#pragma unroll
    for (int rh = 0; rh < C::kHalves; ++rh) {
      const uint32_t cb_ = sb + code_off + rh * (16 * C::kCodeRow);        // rows 16 rh + g and + 8
      const uint32_t sr = sb + C::kScale + (rh * 16 + g) * 16;
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        // lane c's 32 codes of rows g and g + 8 in this 128-wide half: 4 * BITS bytes each
        constexpr uint32_t kMagic = 0x64006400u;
        uint32_t va[4], vb[4];
        const uint32_t ra = cb_ + sub * (16 * BITS), rb = ra + 8 * C::kCodeRow;
        if constexpr (BITS == 3) {
          uint32_t wa[3], wb[3];
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(wa[q]) : "r"(ra + 4 * q));
            asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(wb[q]) : "r"(rb + 4 * q));
          }
          // byte permutes: the two 8-code groups of each 16 in the two 16-bit halves
          va[0] = __byte_perm(wa[0], wa[1], 0x4310); va[1] = __byte_perm(wa[0], wa[1], 0x5421);
          va[2] = __byte_perm(wa[1], wa[2], 0x6532); va[3] = __byte_perm(wa[1], wa[2], 0x7643);
          vb[0] = __byte_perm(wb[0], wb[1], 0x4310); vb[1] = __byte_perm(wb[0], wb[1], 0x5421);
          vb[2] = __byte_perm(wb[1], wb[2], 0x6532); vb[3] = __byte_perm(wb[1], wb[2], 0x7643);
        } else {
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(va[0]), "=r"(va[1]) : "r"(ra));
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(vb[0]), "=r"(vb[1]) : "r"(rb));
          va[2] = va[3] = vb[2] = vb[3] = 0u;
        }
        // pair p as 1024 + code: INT3 codes (16 (p / 8) + m, 16 (p / 8) + m + 8), m = p % 8;
        // INT2 codes (16 (p / 8) + m, + 8) of word p / 8
        auto pair = [&](const uint32_t* v, int p) -> uint32_t {
          const int gq = p >> 3, m = p & 7;
          if constexpr (BITS == 3) {
            const uint32_t w = m < 5 ? v[2 * gq] >> (3 * m) : v[2 * gq + 1] >> (3 * m - 8);
            return lop3_and_or(w, 0x00070007u, kMagic);
          } else {
            return lop3_and_or(v[gq] >> (2 * m), 0x00030003u, kMagic);
          }
        };
        float t[2][4];
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) t[q][e] = tb[sub][q][e];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mma16816(t[j & 1], pair(va, 2 * j), pair(vb, 2 * j), pair(va, 2 * j + 1), pair(vb, 2 * j + 1),
                   bw[sub][2 * j], bw[sub][2 * j + 1]);
        // the scales of this lane's two D columns for rows g and g + 8
        uint32_t h[4];
        asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(h[0]) : "r"(sr + blk_off[sub][0]));
        asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(h[1]) : "r"(sr + blk_off[sub][1]));
        asm volatile("ld.shared.u16 %0, [%1+128];\n" : "=r"(h[2]) : "r"(sr + blk_off[sub][0]));
        asm volatile("ld.shared.u16 %0, [%1+128];\n" : "=r"(h[3]) : "r"(sr + blk_off[sub][1]));
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sc[e] = BF16S ? __uint_as_float(h[e] << 16) : __half2float(__ushort_as_half((uint16_t)h[e]));
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[rh][e] = fmaf(sc[e], t[0][e] + t[1][e], acc[rh][e]);
      }
    }
    if (++slot == C::kRing) { slot = 0; phase ^= 1u; }
    if (++cic < nq && f + 1 < total) continue;

    // ---- this warp's part of the unit is done
    const bool whole = first_cic == 0 && cic == nq;
    bool last = true;
    if (!whole) {
      // parts of this unit: the warps owning its first and last chunk, and those between
      const int item = ei * rgroups + rg;
      const int ux = item * nq;
      const int w0 = ux / L, w1 = (ux + nq - 1) / L;
      // partial slot 0: the piece's first unit; slot 1: its last unit
      float* part = ws.dsplit + ((size_t)wg * 2 + (first_unit ? 0 : 1)) * C::kPart;
#pragma unroll
      for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
        for (int r = 0; r < 4; ++r) part[(rh * 4 + r) * 32 + lane] = acc[rh][r];
      __syncwarp();
      int old = 0;
      if (lane == 0) {
        // release: the warp's partial tile is visible before the ticket moves;
        // acquire: the other parts' tiles are visible to the last arriver
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(ws.dticket + item) : "memory");
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      last = old == w1 - w0;
      if (last) {
        if (lane == 0) ws.dticket[item] = 0;    // free again for fc2 and the next call
        __syncwarp();
        // parts added in chunk order: warps w0 .. w1. Warp w0's piece may begin
        // before the unit (the unit is then its last, slot 1); every later
        // warp's piece begins inside it (slot 0).
        const int hs0 = w0 * L < ux ? 1 : 0;
#pragma unroll
        for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float v = 0.f;
            for (int wk = w0; wk <= w1; ++wk) {
              const int hs = wk == w0 ? hs0 : 0;
              const float pk = wk == wg ? acc[rh][r]
                                        : __ldcg(ws.dsplit + ((size_t)wk * 2 + hs) * C::kPart + (rh * 4 + r) * 32 + lane);
              v = wk == w0 ? pk : v + pk;
            }
            acc[rh][r] = v;
          }
      }
    }
    if (last) {
#pragma unroll
      for (int rh = 0; rh < C::kHalves; ++rh) {
      const int row0 = rg * C::kRows + rh * kRowsPerGroup;
      float v_lo = acc[rh][0] + acc[rh][1];
      float v_hi = acc[rh][2] + acc[rh][3];
      v_lo += __shfl_xor_sync(0xffffffffu, v_lo, 1);
      v_hi += __shfl_xor_sync(0xffffffffu, v_hi, 1);
      if constexpr (FC1) {
        const float up_lo = __shfl_down_sync(0xffffffffu, v_lo, 4);
        const float up_hi = __shfl_down_sync(0xffffffffu, v_hi, 4);
        if ((g & 1) == 0 && (c & 1) == 0 && n < cnt) {
          const int pos = pos0 + n;
          const float sigma = e_scale;
          const float inv = 1.0f / sigma;
          const int j_lo = row0 / 2 + g / 2, j_hi = j_lo + 4;
          const int ex = __ldg(ws.dtab + ei * kDtabInts);
          float2 b_lo = make_float2(0.0f, 0.0f), b_hi = b_lo;
          if (p.b1) {
            b_lo = fc1_bias_pair(p, ex, j_lo);
            b_hi = fc1_bias_pair(p, ex, j_hi);
          }
          const float hs = sigma * sigma * e_hn;
          const float h_lo = silu(v_lo * inv + b_lo.x) * (up_lo * inv + b_lo.y) * hs;
          const float h_hi = silu(v_hi * inv + b_hi.x) * (up_hi * inv + b_hi.y) * hs;
          // fc2 reads these as activations (the 3-bit codes' 16-group permutation)
          ws.h16[(int64_t)pos * p.I + permuted_pos(j_lo, 16)] = __half_as_ushort(__float2half_rn(h_lo));
          ws.h16[(int64_t)pos * p.I + permuted_pos(j_hi, 16)] = __half_as_ushort(__float2half_rn(h_hi));
        }
      } else {
        if ((c & 1) == 0 && n < cnt) {
          const float inv = 1.0f / e_scale;
          const float fct = inv * inv / e_hn * e_w;
          ws.y[(int64_t)e_rid * p.H + row0 + g] = v_lo * fct;
          ws.y[(int64_t)e_rid * p.H + row0 + g + 8] = v_hi * fct;
        }
      }
      }
    }
#pragma unroll
    for (int rh = 0; rh < C::kHalves; ++rh)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[rh][r] = 0.f;
    if (cic == nq) {
      cic = 0;
      if (++rg == rgroups) { rg = 0; ++ei; }
    }
    first_cic = cic;
    first_unit = false;
    fresh = true;
  }
}

template <int ROWS, bool FC1, bool BF16S, bool HAS_ZP>
cudaError_t launch_int4_tma_t(const CUtensorMap& tq, const CUtensorMap& ts, const CUtensorMap& tz,
                              const CUtensorMap& ta, TmaDecodeArgs a, cudaStream_t s) {
  using C = TCfg<ROWS>;
  const cudaError_t err = ensure_smem_optin(decode_int4_tma_kernel<ROWS, FC1, BF16S, HAS_ZP>, (int)C::kSmem);
  if (err != cudaSuccess) return err;
  const int64_t blocks = (int64_t)sm_count() * kTBlocksPerSm;
  return launch_pdl(decode_int4_tma_kernel<ROWS, FC1, BF16S, HAS_ZP>, dim3((unsigned)blocks), dim3(32 * kTWarps), C::kSmem, s, tq, ts, tz, ta, a);
}

// The tensor-copy variant applies when both matmuls' K are multiples of 256 and
// the zero-point rows (if any) are a multiple of 16 bytes long.
// The INT3 / INT2 tensor-copy kernel: implicit zero point, K of both matmuls a multiple of 256.
bool decode_tma23_applies(const Problem& p, bool has_zp) {
  return p.path == QMOE_PATH_DECODE && p.format == QMOE_FORMAT_INT && (p.bits == 3 || p.bits == 2) && !has_zp &&
         p.H % kTChunkK == 0 && p.I % kTChunkK == 0;
}

bool decode_tma_applies(const Problem& p, bool has_zp) {
  if (!decode_int4_blockscaled(p) || p.H % kTChunkK || p.I % kTChunkK) return false;
  return !has_zp || ((p.H / 32) % 16 == 0 && (p.I / 32) % 16 == 0);
}

template <int ROWS, bool FC1>
cudaError_t launch_int4_tma_rows(const uint8_t* q, const uint16_t* scales, const uint8_t* zp, const Problem& p,
                                 const Workspace& ws, cudaStream_t s) {
  const int N = FC1 ? 2 * p.I : p.H, K = FC1 ? p.H : p.I;
  const uint64_t rows = (uint64_t)p.E * N;
  const uint16_t* act = FC1 ? ws.x16 : ws.h16;
  const uint64_t arows = FC1 ? (uint64_t)p.T : (uint64_t)p.R();
  CUtensorMap tq, ts, tz, ta;
  if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, (uint64_t)K / 2, rows, (uint64_t)K / 2, 128,
                   ROWS, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)K / 32, rows, (uint64_t)K / 16, 8,
                   ROWS, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT16, act, (uint64_t)K, arows, (uint64_t)K * 2, kTChunkK, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (zp) {
    if (!make_map_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT8, zp, (uint64_t)K / 32, rows, (uint64_t)K / 32, 16,
                     ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    tz = ts;                                     // not read
  }
  TmaDecodeArgs a{N, K, p, ws};
  const bool bf16 = p.dtype == QMOE_BF16;
  if (bf16) return zp ? launch_int4_tma_t<ROWS, FC1, true, true>(tq, ts, tz, ta, a, s)
                      : launch_int4_tma_t<ROWS, FC1, true, false>(tq, ts, tz, ta, a, s);
  return zp ? launch_int4_tma_t<ROWS, FC1, false, true>(tq, ts, tz, ta, a, s)
            : launch_int4_tma_t<ROWS, FC1, false, false>(tq, ts, tz, ta, a, s);
}

// 32-row units where a unit has at least four chunks (long enough that few of
// them are cut between warps), 16-row units otherwise, and for one or two
// tokens: there the work is a few chunks per warp, and 16-row units give twice
// the warps, each with two chunks in flight (T = 2: 30.9 -> 26.6 us per layer).
template <bool FC1>
cudaError_t launch_int4_tma(const uint8_t* q, const uint16_t* scales, const uint8_t* zp, const Problem& p,
                            const Workspace& ws, cudaStream_t s) {
  const int K = FC1 ? p.H : p.I, N = FC1 ? 2 * p.I : p.H;
  if (p.T > 2 && K / kTChunkK >= 4 && N % 32 == 0) return launch_int4_tma_rows<32, FC1>(q, scales, zp, p, ws, s);
  return launch_int4_tma_rows<16, FC1>(q, scales, zp, p, ws, s);
}


template <int BITS, int ROWS, bool FC1>
cudaError_t launch_int23_tma_rows(const uint8_t* q, const uint16_t* scales, const Problem& p, const Workspace& ws,
                                  cudaStream_t s) {
  using C = T23Cfg<BITS, ROWS>;
  const int N = FC1 ? 2 * p.I : p.H, K = FC1 ? p.H : p.I;
  const uint64_t rows = (uint64_t)p.E * N;
  const uint16_t* act = FC1 ? ws.x16 : ws.h16;
  const uint64_t arows = FC1 ? (uint64_t)p.T : (uint64_t)p.R();
  CUtensorMap tq, ta;
  if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, (uint64_t)K * BITS / 8, rows, (uint64_t)K * BITS / 8,
                   C::kCodeRow, ROWS, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT16, act, (uint64_t)K, arows, (uint64_t)K * 2, kTChunkK, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  Tma23Args a{N, K, p, ws, scales, 31 - __builtin_clz((unsigned)p.block)};
  const bool bf16 = p.dtype == QMOE_BF16;
  const cudaError_t err = bf16 ? ensure_smem_optin(decode_int23_tma_kernel<BITS, ROWS, FC1, true>, (int)C::kSmem)
                               : ensure_smem_optin(decode_int23_tma_kernel<BITS, ROWS, FC1, false>, (int)C::kSmem);
  if (err != cudaSuccess) return err;
  const int64_t blocks = (int64_t)sm_count() * kTBlocksPerSm;
  if (bf16)
    return launch_pdl(decode_int23_tma_kernel<BITS, ROWS, FC1, true>, dim3((unsigned)blocks), dim3(32 * kTWarps),
                      C::kSmem, s, tq, ta, a);
  return launch_pdl(decode_int23_tma_kernel<BITS, ROWS, FC1, false>, dim3((unsigned)blocks), dim3(32 * kTWarps),
                    C::kSmem, s, tq, ta, a);
}

// Unit height as for INT4.
template <int BITS, bool FC1>
cudaError_t launch_int23_tma(const uint8_t* q, const uint16_t* scales, const Problem& p, const Workspace& ws,
                             cudaStream_t s) {
  const int K = FC1 ? p.H : p.I, N = FC1 ? 2 * p.I : p.H;
  if (p.T > 2 && K / kTChunkK >= 4 && N % 32 == 0) return launch_int23_tma_rows<BITS, 32, FC1>(q, scales, p, ws, s);
  return launch_int23_tma_rows<BITS, 16, FC1>(q, scales, p, ws, s);
}

template <bool FC1>
cudaError_t launch_int4_bs(DecodeArgs a, cudaStream_t s) {
  const int64_t blocks = decode_grid_blocks();
  const size_t smem = (size_t)kWarps * kRingB * kSlotBytes;
  const bool bf16 = a.p.dtype == QMOE_BF16, zp = a.zp != nullptr;
  if (bf16) return zp ? launch_int4_bs_t<FC1, true, true>(a, blocks, smem, s)
                      : launch_int4_bs_t<FC1, true, false>(a, blocks, smem, s);
  return zp ? launch_int4_bs_t<FC1, false, true>(a, blocks, smem, s)
            : launch_int4_bs_t<FC1, false, false>(a, blocks, smem, s);
}

int sm_count() { return device_sm_count(); }

template <int BITS, bool FC1, int FMT>
cudaError_t launch_one(DecodeArgs a, int active_max, cudaStream_t s) {
  const int rgroups = a.N / kRowsPerGroup;
  const int64_t items = (int64_t)active_max * rgroups;
  const int64_t warps = (int64_t)sm_count() * kBlocksPerSm * kWarps;
  // the smallest K split that gives every warp several items' worth of chunks
  // Every warp of a team must own at least one K chunk (so that all of them reach
  // the team barriers once per item): ks <= number of 128-wide chunks.
  const int nq = (a.K + kChunkK - 1) / kChunkK;
  int ks = 1;
  while (ks < kWarps && 2 * ks <= nq && items * ks < 4 * warps) ks <<= 1;
  a.ks = ks;
  const int64_t teams_needed = items;
  int64_t blocks = (teams_needed + (kWarps / ks) - 1) / (kWarps / ks);
  const int64_t cap = (int64_t)sm_count() * kBlocksPerSm;
  if (blocks > cap) blocks = cap;
  const size_t smem = (size_t)kWarps * kRing * 2 * 32 * 16 + (size_t)kWarps * 2 * kRing * 32 * 4 +
                      (ks > 1 ? (size_t)(kWarps / ks) * kSlices * 32 * 4 * sizeof(float) : 0);
  const cudaError_t err = ensure_smem_optin(decode_gemv_kernel<BITS, FC1, FMT>, 100 * 1024);
  if (err != cudaSuccess) return err;
  return launch_pdl(decode_gemv_kernel<BITS, FC1, FMT>, dim3((unsigned)blocks), dim3(32 * kWarps), smem, s, a);
}

template <int BITS>
cudaError_t launch_bits(const Problem& p, bool fc1, const uint8_t* q, const void* scales,
                        const uint8_t* zp, const Workspace& ws, cudaStream_t s) {
  const int64_t R = p.R();
  const int active_max = (int)(R < p.E ? R : p.E);
  if constexpr (BITS == 2 || BITS == 3)
    if (decode_tma23_applies(p, zp != nullptr))
      return fc1 ? launch_int23_tma<BITS, true>(q, static_cast<const uint16_t*>(scales), p, ws, s)
                 : launch_int23_tma<BITS, false>(q, static_cast<const uint16_t*>(scales), p, ws, s);
  if (BITS == 4 && decode_tma_applies(p, zp != nullptr))
    return fc1 ? launch_int4_tma<true>(q, static_cast<const uint16_t*>(scales), zp, p, ws, s)
               : launch_int4_tma<false>(q, static_cast<const uint16_t*>(scales), zp, p, ws, s);
  if (BITS == 4 && decode_int4_blockscaled(p)) {
    DecodeArgs a{q, static_cast<const uint16_t*>(scales), zp, fc1 ? ws.x16 : ws.h16,
                 fc1 ? 2 * p.I : p.H, fc1 ? p.H : p.I, 1, p, ws};
    return fc1 ? launch_int4_bs<true>(a, s) : launch_int4_bs<false>(a, s);
  }
  DecodeArgs a{q, static_cast<const uint16_t*>(scales), zp, fc1 ? ws.x16 : ws.h16,
               fc1 ? 2 * p.I : p.H, fc1 ? p.H : p.I, 1, p, ws, fc1 ? p.g1 : p.g2};
  if constexpr (BITS == 4) {
    if (p.format == QMOE_FORMAT_MXFP4)
      return fc1 ? launch_one<4, true, QMOE_FORMAT_MXFP4>(a, active_max, s)
                 : launch_one<4, false, QMOE_FORMAT_MXFP4>(a, active_max, s);
    if (p.format == QMOE_FORMAT_NVFP4)
      return fc1 ? launch_one<4, true, QMOE_FORMAT_NVFP4>(a, active_max, s)
                 : launch_one<4, false, QMOE_FORMAT_NVFP4>(a, active_max, s);
  }
  return fc1 ? launch_one<BITS, true, QMOE_FORMAT_INT>(a, active_max, s)
             : launch_one<BITS, false, QMOE_FORMAT_INT>(a, active_max, s);
}

}  // namespace

int64_t decode_units_max(const Problem& p) {
  // decode-table entries: at most one per expert per pair of routes (<= R, <= E * ceil(T/2))
  int64_t entries = (int64_t)p.E * ((p.T + 1) / 2);
  if (entries > p.R()) entries = p.R();
  return entries * ((2 * p.I > p.H ? 2 * p.I : p.H) / kRowsPerGroup);
}

int64_t decode_split_items_max(const Problem& p) {
  // two partial tiles (the piece's first and last unit) per warp of the grid, in
  // items of 128 floats: one per warp of the cp.async kernel, two (32 rows) per
  // warp of the tensor-copy kernel
  if (!decode_int4_blockscaled(p) && !decode_tma23_applies(p, false)) return 0;
  const int64_t bs = decode_grid_blocks() * kWarps * 2;
  const int64_t tma = (int64_t)sm_count() * kTBlocksPerSm * kTWarps * 2 * (kTPartMax / 128);
  return bs > tma ? bs : tma;
}

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
