// decode_layer.cu -- the decode layer's expert matmuls (T <= 8) as one
// persistent kernel: fc1 dequant-matmul + SwiGLU and fc2 dequant-matmul, the
// weighted fc2 rows left per route for the combine kernel (sm_103a).
//
// Work units: (decode-table entry, 32-row group of the weight matrix, all of K).
// The queue runs through the entries in order and places entry e's fc2 units
// one wave after its fc1 units (after the fc1 units of entries e .. e + D, with
// D fc1-unit lists covering every warp of the grid): by the time an fc2 unit is
// claimed, the fc1 units it needs have normally finished, and the queue ends
// with fc2 units, the small ones. Warps claim units one at a time from a
// counter in the workspace, so warps that stream faster take more units, and
// all finish within about one small unit of each other.
//
// Every warp works on its own: it claims a unit, streams the unit's 256-wide K
// chunks through a private ring of kLStages shared-memory stages with 16-byte
// asynchronous copies (cp.async: each warp instruction moves four rows' 128
// contiguous bytes), and multiplies each chunk as it lands while the next
// chunks are in flight. A stage holds the codes of the unit's 32 weight rows
// for one chunk, their block scales and the chunk's activations of the entry's
// one or two routes. A warp sums a unit's chunks in registers in K order and
// runs the unit's epilogue itself, so no warp waits for another and no partial
// sums cross warps; the copies of the warp's next chunks (of the same or of its
// next unit) stream meanwhile. On this GPU per-lane
// copies from many warps keep more bytes in flight than bulk tensor copies
// issued by one thread (measured 5.1 against 4.4 TB/s on the decode stack's
// weights). The arithmetic of a chunk is the one of decode.cu's block-scaled
// INT4 kernel: codes placed in the FP16 mantissa of 1024, m16n8k16 MMAs whose
// columns are (route, 32-block) pairs, constant MMAs that remove 1024 + zero
// point, block scales applied in FP32 after the MMA.
//
// Shared-memory layout of a stage's codes: [32 rows][128 B], each row's 16-byte
// pieces XOR-swizzled by 4 (row mod 2), so the two rows that a quarter of a
// warp reads at once (rows g and g + 1) land in opposite halves of the banks.
//
// fc1 epilogue: h = silu(gate) * up from the interleaved rows 2j / 2j+1
// (activation_type "swiglu", swiglu_fusion = 1), stored in FP16 with the
// token's power of two squared, as decode.cu does; then the unit counts itself
// done for its entry (a release reduction). An fc2 unit's activations are
// copied only once all fc1 units of its entry are counted. A warp that would
// have to wait for them first finishes every chunk it has in flight, so a
// waiting warp holds no started unit and its claimed ones lie later in the
// queue; every fc1 unit precedes the fc2 units of its entry in the queue, so
// the wait always ends. fc2 epilogue: y = (W2 h)
// / scale^2 * w_route in FP32 per route id, stored without waiting; combine.cu
// then sums each token's routes. The result depends neither on which warp takes
// which unit nor on the batch.
//
// Every wait is bounded (1 s). A warp that gives up sets the error flag in the
// workspace counters, which makes the combine kernel write NaN to the output,
// lets its copies in flight land and stops.
#include "tma.cuh"
#include <cuda_fp8.h>

namespace qmoe {
namespace {

constexpr int kLWarps = 4;                           // warps per block, each on its own units
constexpr int kLThreads = 32 * kLWarps;
constexpr int kLRows = 32;                           // weight rows per unit
constexpr int kLChunk = 256;                         // K per stage
constexpr int kLStages = 3;                          // ring depth of a warp
constexpr int kLBlocksPerSm = 3;                     // resident blocks per SM (registers, shared memory)
constexpr int kLCodes = kLRows * 128;                // [32 rows][128 B], swizzled
constexpr int kLScale = kLCodes;                     // [32 rows][8] 16-bit scales
constexpr int kLAct = kLScale + kLRows * 16;         // [2 routes][256] FP16
constexpr int kLStage = kLAct + 2 * 512;
constexpr int kLRingBytes = kLStages * kLStage;      // one warp's ring
constexpr int kLZeroOff = kLWarps * kLRingBytes + 32;   // 32 mod 128
constexpr int kLZero = 512;                          // zeros read by lanes with no activations
constexpr int kLMetaOff = kLZeroOff + kLZero + 96;   // [warp][stage] int4, 16-byte aligned
constexpr int kLReadyOff = kLMetaOff + kLWarps * kLStages * 16;   // [kDtabMax / 32] entries whose fc1 is done
constexpr int kLDtabOff = kLReadyOff + kDtabMax / 8;              // the decode table, [entries][kDtabInts]
constexpr int kLSmemFixed = 128 + kLDtabOff;                      // + the decode table's bytes
constexpr uint64_t kLWaitNs = QMOE_WAIT_LIMIT_NS;
constexpr int kErrLayerTimeout = 3;
static_assert(kLStage % 128 == 0, "stages keep the code rows 128-byte aligned");
static_assert(kLZeroOff % 128 == 32, "the zero area must not share banks with the activation tiles");
static_assert(kLMetaOff % 16 == 0 && kLDtabOff % 16 == 0, "vector accesses");

struct LayerArgs {
  Problem p;
  Workspace ws;
  const uint8_t* q1;       // fc1 codes [E][2I][H/2]
  const uint16_t* s1;      // fc1 scales [E][2I][H/32]
  const uint8_t* q2;       // fc2 codes [E][H][I/2]
  const uint16_t* s2;      // fc2 scales [E][H][I/32]
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Wait until at most n of this thread's committed copy groups are still in flight.
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  static_assert(kLStages <= 8, "one case per possible count");
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;\n" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;\n" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;\n" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;\n" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;\n" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;\n" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;\n" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;\n" ::: "memory"); break;
  }
}

__device__ __forceinline__ int ld_acquire(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void red_add_release(int* ptr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(ptr), "r"(v) : "memory");
}

// The block's record of entries whose fc1 units are all done: set by the warp
// that saw the count complete (after its acquire), read by the others with
// block-scope acquire, so their copies of the entry's h16 follow that acquire.
__device__ __forceinline__ void ready_set(uint32_t* word, uint32_t bit) {
  asm volatile("red.release.cta.shared::cta.or.b32 [%0], %1;\n" ::"r"(smem_u32(word)), "r"(bit) : "memory");
}
__device__ __forceinline__ uint32_t ready_get(const uint32_t* word) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];\n" : "=r"(v) : "r"(smem_u32(word)) : "memory");
  return v;
}

// ---- FP4 expert formats (E2M1 codes, 8-bit block scales; see qmoe.h)
// Byte r of w (codes 2r and 2r + 1) as an FP16 pair: the low half from the low
// nibble (the hardware conversion, exact: every E2M1 value is an FP16 value).
__device__ __forceinline__ uint32_t e2m1x2(uint32_t w, int r) {
  const uint32_t b = (w >> (8 * r)) & 0xFFu;
  uint32_t h;
  asm("{\n .reg .b8 q;\n cvt.u8.u32 q, %1;\n cvt.rn.f16x2.e2m1x2 %0, q;\n}\n" : "=r"(h) : "r"(b));
  return h;
}

// E8M0 block scale 2^(b - 127) as an FP32 value (exact; 255 is NaN).
__device__ __forceinline__ float e8m0_value(uint32_t b) {
  if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
  return b == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// E4M3 block scale as an FP16 pair (exact in FP16).
__device__ __forceinline__ uint32_t e4m3_half2(uint32_t b) {
  const uint32_t h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3).x;
  return h | (h << 16);
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src) : "memory");
}

// Unit q of the queue: the fc1 units (a per entry) of entries 0 .. L-1, then
// rounds r = L .. entries-1 of entry r's fc1 units followed by entry r-L's fc2
// units (b per entry), then the fc2 units of the last L entries.
struct UnitQueue {
  int entries, a, b, L;
  __device__ __forceinline__ void decode(int q, bool& f1, int& ei, int& rg) const {
    const int p1 = L * a, p2 = p1 + (entries - L) * (a + b);
    if (q < p1) {
      f1 = true;
      ei = q / a;
      rg = q - ei * a;
    } else if (q < p2) {
      const int q2 = q - p1, r = q2 / (a + b), o = q2 - r * (a + b);
      f1 = o < a;
      ei = f1 ? L + r : r;
      rg = f1 ? o : o - a;
    } else {
      const int q3 = q - p2, r = q3 / b;
      f1 = false;
      ei = entries - L + r;
      rg = q3 - r * b;
    }
  }
};

template <bool BF16S, int FMT>
__global__ void __launch_bounds__(kLThreads, kLBlocksPerSm) decode_layer_kernel(LayerArgs a) {
  constexpr bool kFp4 = FMT != QMOE_FORMAT_INT;
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* base = smem + ((128u - (smem_u32(smem) & 127u)) & 127u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring_s = smem_u32(base) + warp * kLRingBytes;
  const uint32_t zero_s = smem_u32(base) + kLZeroOff;
  int4* const meta = reinterpret_cast<int4*>(base + kLMetaOff) + warp * kLStages;
  uint32_t* const s_ready = reinterpret_cast<uint32_t*>(base + kLReadyOff);
  int* const s_dtab = reinterpret_cast<int*>(base + kLDtabOff);
  if (threadIdx.x < kLZero / 4) reinterpret_cast<uint32_t*>(base + kLZeroOff)[threadIdx.x] = 0u;
  if (threadIdx.x < kDtabMax / 32) s_ready[threadIdx.x] = 0u;
  // routing, the decode table, x16 and the zeroed synchronisation words come
  // from the routing kernel
  pdl_wait();
  pdl_trigger();

  int* const claim = ws.dsync;
  int* const fc1_done = ws.dsync + kSyncHeader;
  const int entries = ws.counters[3];
  // the warp's first claim is in flight while the block copies the decode table
  int first_unit = 0;
  if (lane == 0) first_unit = atomicAdd(claim, 1);
  for (int i = threadIdx.x * 4; i < entries * kDtabInts; i += blockDim.x * 4)
    *reinterpret_cast<int4*>(s_dtab + i) = __ldg(reinterpret_cast<const int4*>(ws.dtab + i));
  __syncthreads();

  const int N1 = 2 * p.I, N2 = p.H;
  const int rg1 = N1 / kLRows, rg2 = N2 / kLRows;
  const int nunits = entries * (rg1 + rg2);
  // the lag L (in entries) puts an entry's fc2 units at least one wave of claims
  // (one unit per warp) after its last fc1 unit
  int lag = (int)(gridDim.x * kLWarps) / rg1 + 2;
  if (lag > entries) lag = entries;
  const UnitQueue queue{entries, rg1, rg2, lag};
  const int nst1 = p.H / kLChunk, nst2 = p.I / kLChunk;

  // ---- issue side: the unit whose chunks are being copied, and the claim after it
  int iu = __shfl_sync(0xffffffffu, first_unit, 0);
  // the warp's next unit is claimed (lane 0) when the copies of the current
  // unit's last two chunks are issued: late enough that units go to the warps
  // that free up first, early enough to hide the atomic's round trip
  int next = nunits;
  int ij = 0, inst = 0, iK = 0, icnt = 0, ia0 = 0, ia1 = 0, iei = 0;
  bool if1 = true, iready = true;
  const uint8_t* iq = nullptr;
  const uint8_t* is = nullptr;
  const uint8_t* iact = nullptr;
  auto start_unit = [&](int u) {
    int rg;
    queue.decode(u, if1, iei, rg);
    const int* d = s_dtab + iei * kDtabInts;
    const int row0 = d[0] * (if1 ? N1 : N2) + rg * kLRows;
    icnt = d[2];
    ia0 = if1 ? d[4] : d[1];
    ia1 = if1 ? d[5] : d[1] + 1;
    inst = if1 ? nst1 : nst2;
    iK = if1 ? p.H : p.I;
    iq = (if1 ? a.q1 : a.q2) + (int64_t)row0 * (iK / 2);
    // a row's scales: K/32 16-bit ones (INT4), K/32 E8M0 bytes, K/16 E4M3 bytes
    is = reinterpret_cast<const uint8_t*>(if1 ? a.s1 : a.s2) +
         (int64_t)row0 * (FMT == QMOE_FORMAT_MXFP4 ? iK / 32 : iK / 16);
    iact = reinterpret_cast<const uint8_t*>(if1 ? ws.x16 : ws.h16);
    ij = 0;
    iready = if1;
  };
  if (iu < nunits) start_unit(iu);

  // ---- compute side
  const int g = lane >> 2, c = lane & 3;
  const bool owner = (g & 3) == c;               // supplies the activations of MMA column g
  const int on = g >> 2;                         // that column's route within the entry
  const int n = c >> 1;                          // route of this lane's D columns
  // this lane's 16-byte code pieces of row g: logical piece c (first 128 K) and
  // c + 4 (second), swizzled by 4 (g mod 2)
  const uint32_t code_off = (uint32_t)g * 128 + ((uint32_t)(c ^ (4 * (g & 1))) << 4);
  const uint32_t scale_off = kLScale + (uint32_t)g * 16 + 4u * (c & 1);
  const uint32_t act_off = (uint32_t)(kLAct + on * 512 + 64 * c);

  const __half2 ne_d = __float2half2_rn(-(1024.0f + 8.0f)), no_d = __float2half2_rn(-(1024.0f + 128.0f));
  const uint32_t ne_def = *reinterpret_cast<const uint32_t*>(&ne_d);
  const uint32_t no_def = *reinterpret_cast<const uint32_t*>(&no_d);
  constexpr uint32_t kMagic = 0x64006400u;

  float acc[2][4];
  bool f1 = true;
  int ei = 0, rg = 0, cnt = 0, pos0 = 0, ex = 0, e_rid = 0;
  float e_scale = 1.0f, e_w = 0.0f, e_hn = 1.0f;
  int issued = 0, computed = 0;
  bool ok = true;

  for (;;) {
    // ---- issue: keep up to kLStages chunks in flight
    while (ok && iu < nunits && issued - computed < kLStages) {
      if (!iready) {
        // an fc2 unit's activations are its entry's SwiGLU outputs: every fc1
        // unit of the entry has stored its h16 values
        uint32_t* word = s_ready + (iei >> 5);
        const uint32_t bit = 1u << (iei & 31);
        if (!(ready_get(word) & bit)) {
          int done = 0;
          if (lane == 0) done = ld_acquire(fc1_done + iei) >= rg1;
          done = __shfl_sync(0xffffffffu, done, 0);
          if (!done) {
            // finish the chunks in flight first: a waiting warp holds no unfinished unit
            if (issued != computed) break;
            int good = 1;
            if (lane == 0) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire(fc1_done + iei) < rg1) {
                if (globaltimer_ns() - t0 >= kLWaitNs) { good = 0; break; }
                __nanosleep(128);
              }
            }
            if (!__shfl_sync(0xffffffffu, good, 0)) {
              if (lane == 0) atomicExch(ws.counters + 2, kErrLayerTimeout);
              ok = false;
              break;
            }
          }
          if (lane == 0) ready_set(word, bit);
          __syncwarp();                          // the other lanes' copies follow lane 0's acquire
        }
        iready = true;
      }
      const int st = issued % kLStages;
      const uint32_t sb = ring_s + st * kLStage;
      // codes: instruction i copies rows 4 i .. 4 i + 3, 128 bytes each
      {
        const int r0 = lane >> 3, pc = lane & 7;
        const uint32_t dst = sb + r0 * 128 + ((uint32_t)(pc ^ (4 * (r0 & 1))) << 4);
        const uint8_t* src = iq + (int64_t)r0 * (iK / 2) + ij * 128 + pc * 16;
#pragma unroll
        for (int i = 0; i < kLRows / 4; ++i) cp_async16(dst + i * 512, src + (int64_t)i * 4 * (iK / 2));
      }
      // scales: row `lane`'s scales of the chunk: 8 16-bit ones, 8 E8M0 bytes
      // (MXFP4) or 16 E4M3 bytes (NVFP4)
      if constexpr (FMT == QMOE_FORMAT_MXFP4)
        cp_async8(sb + kLScale + lane * 16, is + (int64_t)lane * (iK / 32) + ij * 8);
      else
        cp_async16(sb + kLScale + lane * 16, is + (int64_t)lane * (iK / 16) + ij * 16);
      // activations: [route][256] FP16
      cp_async16(sb + kLAct + lane * 16, iact + (int64_t)ia0 * iK * 2 + ij * 512 + lane * 16);
      if (icnt > 1) cp_async16(sb + kLAct + 512 + lane * 16, iact + (int64_t)ia1 * iK * 2 + ij * 512 + lane * 16);
      cp_async_commit();
      if (lane == 0) {
        meta[st] = make_int4(iu, ij, inst, 0);
        if (ij == (inst > 2 ? inst - 2 : 0)) next = atomicAdd(claim, 1);
      }
      ++issued;
      if (++ij == inst) {
        iu = __shfl_sync(0xffffffffu, next, 0);
        if (iu < nunits) start_unit(iu);
      }
    }
    if (issued == computed) break;               // no work left, or a wait gave up

    // ---- compute the oldest chunk in flight
    cp_async_wait_pending(issued - computed - 1);
    __syncwarp();
    const int st = computed % kLStages;
    const int4 m = meta[st];
    const int u = m.x, j = m.y, nst = m.z;
    const uint32_t sb = ring_s + st * kLStage;
    if (j == 0) {
      queue.decode(u, f1, ei, rg);
      const int* d = s_dtab + ei * kDtabInts;
      ex = d[0];
      pos0 = d[1];
      cnt = d[2];
      e_hn = __int_as_float(d[7]);   // the expert's SwiGLU normalisation
      e_rid = n ? d[6] : d[3];
      if (n < cnt) {
        e_scale = __ldg(ws.tok_scale + (n ? d[5] : d[4]));
        if (!f1) e_w = __ldg(ws.topk_w + e_rid);
      }
#pragma unroll
      for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[rh][r] = 0.f;
    }
    {
      const uint32_t ab = owner ? sb + act_off : zero_s;
      // activations (B fragments) of both 128-wide halves, shared by both row halves
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
      // the implicit zero point gives every row the same bias operand: its MMAs
      // run once per chunk, in chains of their own, and join both row halves' sums
      float tb[2][2][4];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) tb[sub][q][e] = 0.f;
      if constexpr (!kFp4) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            mma16816(tb[sub][0], ne_def, ne_def, no_def, no_def, bw[sub][4 * i], bw[sub][4 * i + 1]);
            mma16816(tb[sub][1], ne_def, ne_def, no_def, no_def, bw[sub][4 * i + 2], bw[sub][4 * i + 3]);
          }
      }
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        // rows 16 rh + g and 16 rh + 8 + g share the swizzle term, so the second
        // is 8 row pitches further
        const uint32_t cb = sb + code_off + rh * (16 * 128);
        const uint32_t sr = sb + scale_off + rh * (16 * 16);
        uint4 cw[2][2];
        uint32_t sw[2][2];
        // piece c + 4 sits 64 bytes away from piece c in the other half of the row
        const uint32_t cb1 = cb ^ 64u;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(cw[0][0].x), "=r"(cw[0][0].y), "=r"(cw[0][0].z), "=r"(cw[0][0].w) : "r"(cb));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+1024];\n"
                     : "=r"(cw[0][1].x), "=r"(cw[0][1].y), "=r"(cw[0][1].z), "=r"(cw[0][1].w) : "r"(cb));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(cw[1][0].x), "=r"(cw[1][0].y), "=r"(cw[1][0].z), "=r"(cw[1][0].w) : "r"(cb1));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+1024];\n"
                     : "=r"(cw[1][1].x), "=r"(cw[1][1].y), "=r"(cw[1][1].z), "=r"(cw[1][1].w) : "r"(cb1));
        if constexpr (FMT == QMOE_FORMAT_INT) {
          asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(sw[0][0]) : "r"(sr));
          asm volatile("ld.shared.u32 %0, [%1+128];\n" : "=r"(sw[0][1]) : "r"(sr));
          asm volatile("ld.shared.u32 %0, [%1+8];\n" : "=r"(sw[1][0]) : "r"(sr));
          asm volatile("ld.shared.u32 %0, [%1+136];\n" : "=r"(sw[1][1]) : "r"(sr));
        } else {
          // MXFP4: the E8M0 bytes of this lane's two block columns (blocks 2 (c & 1)
          // and +1 of each half); NVFP4: the E4M3 bytes of the two 16-wide blocks of
          // each of the lane's code pieces (pieces c and c + 4)
          const uint32_t srow = sb + kLScale + (uint32_t)(rh * 16 + g) * 16;
          const uint32_t o0 = FMT == QMOE_FORMAT_MXFP4 ? 2u * (c & 1) : 2u * c;
          const uint32_t o1 = FMT == QMOE_FORMAT_MXFP4 ? 4u + 2u * (c & 1) : 8u + 2u * c;
          asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(sw[0][0]) : "r"(srow + o0));
          asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(sw[0][1]) : "r"(srow + 8 * 16 + o0));
          asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(sw[1][0]) : "r"(srow + o1));
          asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(sw[1][1]) : "r"(srow + 8 * 16 + o1));
        }
        float t[2][2][4];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub)
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) t[sub][q][e] = 0.f;
        if constexpr (!kFp4) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
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
        } else {
          // E2M1 pairs straight from the codes: byte r of a word holds codes 2r and
          // 2r + 1, which one conversion turns into an FP16 pair (activations in
          // natural K order); NVFP4 multiplies each word's pairs by the E4M3 scale
          // of its 16-wide block (words 0-1 and 2-3 of a piece) before the MMA
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const uint32_t wa = (&cw[sub][0].x)[i], wb = (&cw[sub][1].x)[i];
              uint32_t a0 = e2m1x2(wa, 0), a1 = e2m1x2(wb, 0), a2 = e2m1x2(wa, 1), a3 = e2m1x2(wb, 1);
              uint32_t a4 = e2m1x2(wa, 2), a5 = e2m1x2(wb, 2), a6 = e2m1x2(wa, 3), a7 = e2m1x2(wb, 3);
              if constexpr (FMT == QMOE_FORMAT_NVFP4) {
                const uint32_t sa = e4m3_half2((sw[sub][0] >> (8 * (i >> 1))) & 0xFFu);
                const uint32_t sbv = e4m3_half2((sw[sub][1] >> (8 * (i >> 1))) & 0xFFu);
                a0 = hmul2_bits(a0, sa); a2 = hmul2_bits(a2, sa); a4 = hmul2_bits(a4, sa); a6 = hmul2_bits(a6, sa);
                a1 = hmul2_bits(a1, sbv); a3 = hmul2_bits(a3, sbv); a5 = hmul2_bits(a5, sbv); a7 = hmul2_bits(a7, sbv);
              }
              mma16816(t[sub][0], a0, a1, a2, a3, bw[sub][4 * i], bw[sub][4 * i + 1]);
              mma16816(t[sub][1], a4, a5, a6, a7, bw[sub][4 * i + 2], bw[sub][4 * i + 3]);
            }
        }
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          float s_a0, s_a1, s_b0, s_b1;
          const uint32_t swa = sw[sub][0], swb = sw[sub][1];
          if constexpr (FMT == QMOE_FORMAT_MXFP4) {
            s_a0 = e8m0_value(swa & 0xFFu); s_a1 = e8m0_value((swa >> 8) & 0xFFu);
            s_b0 = e8m0_value(swb & 0xFFu); s_b1 = e8m0_value((swb >> 8) & 0xFFu);
          } else if constexpr (FMT == QMOE_FORMAT_NVFP4) {
            s_a0 = s_a1 = s_b0 = s_b1 = 1.0f;       // applied before the MMA
          } else if constexpr (BF16S) {
            s_a0 = __uint_as_float(swa << 16); s_a1 = __uint_as_float(swa & 0xFFFF0000u);
            s_b0 = __uint_as_float(swb << 16); s_b1 = __uint_as_float(swb & 0xFFFF0000u);
          } else {
            s_a0 = __half2float(__ushort_as_half((uint16_t)(swa & 0xFFFFu)));
            s_a1 = __half2float(__ushort_as_half((uint16_t)(swa >> 16)));
            s_b0 = __half2float(__ushort_as_half((uint16_t)(swb & 0xFFFFu)));
            s_b1 = __half2float(__ushort_as_half((uint16_t)(swb >> 16)));
          }
          const float s4[4] = {s_a0, s_a1, s_b0, s_b1};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[rh][e] = fmaf(s4[e], (t[sub][0][e] + t[sub][1][e]) + (tb[sub][0][e] + tb[sub][1][e]), acc[rh][e]);
        }
      }
    }
    // every lane's shared-memory reads of the stage are done before it is refilled
    __syncwarp();
    ++computed;
    if (j + 1 < nst) continue;

    // ---- the unit's last chunk: its epilogue
    float v[2][2];                               // [row half][row g, row g + 8], route n
    // NVFP4: the expert's global scale of this matmul
    const float* gsc = f1 ? p.g1 : p.g2;
    const float gf = (FMT == QMOE_FORMAT_NVFP4 && gsc) ? __ldg(gsc + ex) : 1.0f;
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      v[rh][0] = acc[rh][0] + acc[rh][1];
      v[rh][1] = acc[rh][2] + acc[rh][3];
      v[rh][0] += __shfl_xor_sync(0xffffffffu, v[rh][0], 1);
      v[rh][1] += __shfl_xor_sync(0xffffffffu, v[rh][1], 1);
      v[rh][0] *= gf;
      v[rh][1] *= gf;
    }
    if (f1) {
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        // gate rows 2j sit at even MMA rows g, their up rows at g + 1
        const float up_lo = __shfl_down_sync(0xffffffffu, v[rh][0], 4);
        const float up_hi = __shfl_down_sync(0xffffffffu, v[rh][1], 4);
        if ((g & 1) == 0 && (c & 1) == 0 && n < cnt) {
          const int hp = pos0 + n;
          const float sigma = e_scale;
          const float inv = 1.0f / sigma;
          const int j_lo = (rg * kLRows + 16 * rh + g) / 2, j_hi = j_lo + 4;
          float2 b_lo = make_float2(0.0f, 0.0f), b_hi = b_lo;
          if (p.b1) {
            b_lo = fc1_bias_pair(p, ex, j_lo);
            b_hi = fc1_bias_pair(p, ex, j_hi);
          }
          const float hs = sigma * sigma * e_hn;
          const float h_lo = silu(v[rh][0] * inv + b_lo.x) * (up_lo * inv + b_lo.y) * hs;
          const float h_hi = silu(v[rh][1] * inv + b_hi.x) * (up_hi * inv + b_hi.y) * hs;
          // fc2 reads these as activations: for INT4 K-order permuted, odd K
          // positions carrying 1/16
          const int pj0 = (j_lo & ~7) + ((j_lo & 7) < 4 ? 2 * (j_lo & 7) : 2 * (j_lo & 7) - 7);
          const int pj1 = (j_hi & ~7) + ((j_hi & 7) < 4 ? 2 * (j_hi & 7) : 2 * (j_hi & 7) - 7);
          if constexpr (kFp4) {
            // natural K order, plain values (the FP4 operand pairs are adjacent codes)
            ws.h16[(int64_t)hp * p.I + j_lo] = __half_as_ushort(__float2half_rn(h_lo));
            ws.h16[(int64_t)hp * p.I + j_hi] = __half_as_ushort(__float2half_rn(h_hi));
          } else {
            ws.h16[(int64_t)hp * p.I + pj0] = __half_as_ushort(__float2half_rn((j_lo & 1) ? h_lo * 0.0625f : h_lo));
            ws.h16[(int64_t)hp * p.I + pj1] = __half_as_ushort(__float2half_rn((j_hi & 1) ? h_hi * 0.0625f : h_hi));
          }
        }
      }
      // publish: the unit's h16 values are stored (the release orders the
      // other lanes' stores, which the warp barrier ordered before it)
      __syncwarp();
      if (lane == 0) red_add_release(fc1_done + ei, 1);
    } else {
      const float inv = 1.0f / e_scale;
      const float fct = inv * inv / e_hn * e_w;
      if ((c & 1) == 0 && n < cnt) {
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          const int row = rg * kLRows + 16 * rh + g;
          __stcg(ws.y + (int64_t)e_rid * p.H + row, v[rh][0] * fct);
          __stcg(ws.y + (int64_t)e_rid * p.H + row + 8, v[rh][1] * fct);
        }
      }
    }
  }
  // this lane's copies in flight (none unless a wait gave up) land before the
  // block's shared memory is released
  cp_async_wait_all();
}

}  // namespace

bool decode_layer_applies(const Problem& p, bool has_zp) {
  const bool fmt_ok = (p.format == QMOE_FORMAT_INT && p.block == 32) ||
                      (p.format == QMOE_FORMAT_MXFP4 && p.block == 32) ||
                      (p.format == QMOE_FORMAT_NVFP4 && p.block == 16);
  return !has_zp && p.path == QMOE_PATH_DECODE && fmt_ok && p.bits == 4 && p.T <= kDecodeMaxT &&
         p.H % kLChunk == 0 && p.I % kLChunk == 0;
}

cudaError_t launch_decode_layer(const Problem& p, const uint8_t* fc1_q, const void* fc1_scales,
                                const uint8_t* fc2_q, const void* fc2_scales, const Workspace& ws,
                                cudaStream_t s) {
  LayerArgs a{p, ws, fc1_q, static_cast<const uint16_t*>(fc1_scales), fc2_q,
              static_cast<const uint16_t*>(fc2_scales)};
  // the decode table's share of shared memory is sized by the entries it can hold
  int64_t entries = (int64_t)p.E * ((p.T + 1) / 2);
  if (entries > p.R()) entries = p.R();
  const size_t smem = (size_t)kLSmemFixed + (size_t)entries * kDtabInts * 4;
  int per_sm = (int)((228 * 1024) / (smem + 1024));
  if (per_sm > kLBlocksPerSm) per_sm = kLBlocksPerSm;
  if (per_sm < 1) return cudaErrorNotSupported;
  // one block short of filling every SM: the next layer's routing block (a
  // single block with little shared memory) finds room at once and routes while
  // this kernel runs
  const int blocks = device_sm_count() * per_sm - 1;
  auto go = [&](auto kernel) -> cudaError_t {
    const cudaError_t err = ensure_smem_optin(kernel, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kernel, dim3(blocks), dim3(kLThreads), smem, s, a);
  };
  // the FP4 formats' scales are 8-bit, so the activation dtype plays no part there
  if (p.format == QMOE_FORMAT_MXFP4) return go(decode_layer_kernel<false, QMOE_FORMAT_MXFP4>);
  if (p.format == QMOE_FORMAT_NVFP4) return go(decode_layer_kernel<false, QMOE_FORMAT_NVFP4>);
  if (p.dtype == QMOE_BF16) return go(decode_layer_kernel<true, QMOE_FORMAT_INT>);
  return go(decode_layer_kernel<false, QMOE_FORMAT_INT>);
}

}  // namespace qmoe
