// decode_layer.cu -- the decode layer (T <= 8) after routing as one persistent
// kernel: fc1 dequant-matmul + SwiGLU, fc2 dequant-matmul and the
// routing-weighted combine (sm_103a).
//
// Work units: (decode-table entry, 32-row group of the weight matrix, all of K),
// first every fc1 unit, then every fc2 unit, each list in entry order. Blocks
// claim units one at a time from a counter in the workspace, so blocks that
// stream faster take more units, and all finish within about one small unit of
// each other.
//
// Each block (three per SM) has one producer warp and four consumer warps
// around a ring of shared-memory slots. A slot holds a group of four 256-wide K
// chunks of one unit, brought in by three or four bulk tensor copies: the codes
// of the unit's 32 weight rows for the four chunks (one 3-D box, 128-byte
// swizzle), their block scales (one 3-D box) and the chunks' activations of the
// entry's one or two routes (one 2-D box per route). Few, large copies keep the
// producer's issue cost per byte low. Consumer warp w multiplies chunk w of
// every slot, so a unit's chunks are multiplied side by side and every warp
// sees every phase of every slot's barriers. A warp sums its chunks of a unit in
// registers, in K order; the warp that finishes the unit's last chunk adds the
// warps' sums in K order (warp position 0, 1, 2, 3 of the unit) and runs the
// epilogue. The arithmetic of a chunk is the one of decode.cu's block-scaled
// INT4 kernel: codes placed in the FP16 mantissa of 1024, m16n8k16 MMAs whose
// columns are (route, 32-block) pairs, constant MMAs that remove 1024 + zero
// point, block scales applied in FP32 after the MMA.
//
// Shared-memory layout of a slot's codes: [32 rows][4 chunks][128 B]; the
// swizzle XORs a row's 16-byte pieces with bits 7-9 of their address, i.e. with
// (4 row + chunk) mod 8, so the two rows that a quarter of a warp reads at once
// (rows g and g + 1 of one chunk) land in opposite halves of the banks.
//
// fc1 epilogue: h = silu(gate) * up from the interleaved rows 2j / 2j+1
// (activation_type "swiglu", swiglu_fusion = 1), stored in FP16 with the
// token's power of two squared, as decode.cu does; then the unit counts itself
// done for its entry. An fc2 unit's activations are copied in only once all fc1
// units of its entry are counted; its weights are copied before that. The fc1
// units were all claimed earlier by running blocks, which never wait on fc2
// work, so the wait always ends. fc2 epilogue: y = (W2 h) / scale^2 * w_route in
// FP32 per route id; then, per (token, 32-row group of H), the unit that brings
// the last of the token's k routes adds the k rows in j order, rounds once and
// writes the output: the sum and the rounding of combine.cu ("[CUDA] Add
// MoEPacked CPU/GPU hybrid offload ..." #33973: FP32 partial sum rounded once,
// NaN kept, zero-weight routes skipped; FC2 bias per route before the rounding,
// "[CUDA] Add INT4 and INT3 QMoE CPU/GPU offload support" #33575). The result
// depends neither on which block takes which unit nor on the batch.
//
// Every wait is bounded (1 s). A warp that gives up sets the error flag in the
// workspace counters; the producer then waits (bounded) for its copies in
// flight; the last block to finish fills the output with NaN when the flag is
// set, so a failed call never returns plausible numbers.
#include "tma.cuh"

namespace qmoe {
namespace {

constexpr int kLConsumers = 4;                       // consumer warps
constexpr int kLThreads = 32 * (kLConsumers + 1);    // + one producer warp
constexpr int kLRows = 32;                           // weight rows per unit
constexpr int kLChunk = 256;                         // K per chunk
constexpr int kLGroup = kLConsumers;                 // chunks per slot: one per consumer warp
constexpr int kLRing = 3;                            // slots per block
constexpr int kLUnitSlots = 4;                       // units whose partial sums a block holds
constexpr int kLCodes = kLRows * kLGroup * 128;      // [32 rows][4 chunks][128 B], swizzled
constexpr int kLScale = kLCodes;                     // [32 rows][4 chunks][8] 16-bit scales
constexpr int kLAct = kLScale + kLRows * kLGroup * 16;   // [2 routes][4 chunks][256] FP16
constexpr int kLSlot = kLAct + 2 * kLGroup * 512;
constexpr int kLPartOff = kLRing * kLSlot;           // [unit slot][warp position][4][16] FP32
constexpr int kLZeroOff = kLPartOff + kLUnitSlots * kLConsumers * 64 * 4 + 32;   // 32 mod 128
constexpr int kLZero = 512;                          // zeros read by lanes with no activations
constexpr int kLBarOff = kLZeroOff + kLZero + 96;    // 8-byte aligned
constexpr int kLMetaOff = kLBarOff + 2 * kLRing * 8;          // [kLRing] int4
constexpr int kLUnitOff = kLMetaOff + kLRing * 16;            // [kLUnitSlots] arrivals, done sequence
constexpr int kLFlagOff = kLUnitOff + 2 * kLUnitSlots * 4;
constexpr int kLReadyOff = kLFlagOff + 16;                   // [kDtabMax / 32] entries whose fc1 is done
constexpr int kLDtabOff = kLReadyOff + kDtabMax / 8;         // the decode table, [entries][kDtabInts]
constexpr int kLSmemFixed = 1024 + kLDtabOff;                // + the decode table's bytes
constexpr uint64_t kLWaitNs = 1000000000ull;         // 1 s: far beyond any legitimate wait
constexpr uint64_t kLDrainNs = 100000000ull;
constexpr int kErrLayerTimeout = 3;
static_assert(kLSlot % 1024 == 0, "swizzled code tiles need 1024-byte aligned slots");
static_assert(kLZeroOff % 128 == 32, "the zero area must not share banks with the activation tiles");
static_assert(kLMetaOff % 16 == 0 && kLDtabOff % 16 == 0, "vector accesses");

struct LayerArgs {
  Problem p;
  Workspace ws;
  uint16_t* out;
};

__device__ __forceinline__ int ld_acquire(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ int atom_add_acq_rel(int* ptr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(int* ptr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(ptr), "r"(v) : "memory");
}

// The generic-proxy writes this thread has acquired become visible to its
// following bulk tensor copies.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

// Consumer wait on a chunk: bounded, and ends early when the producer gave up.
__device__ __forceinline__ bool consumer_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && (*abort || globaltimer_ns() - t0 > kLWaitNs)) return false;
  }
}

// Bounded wait until a shared word reaches `want`.
__device__ __forceinline__ bool smem_wait_eq(const volatile int* word, int want) {
  if (*word == want) return true;
  const uint64_t t0 = globaltimer_ns();
  while (*word != want) {
    if (globaltimer_ns() - t0 > kLWaitNs) return false;
    __nanosleep(32);
  }
  return true;
}

template <bool BF16S>
__global__ void __launch_bounds__(kLThreads, 3) decode_layer_kernel(
    const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap ts1,
    const __grid_constant__ CUtensorMap tq2, const __grid_constant__ CUtensorMap ts2,
    const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap th, LayerArgs a) {
  const Problem& p = a.p;
  const Workspace& ws = a.ws;
  extern __shared__ __align__(16) uint8_t smem[];
  // the swizzled code tiles need 1024-byte aligned destinations
  uint8_t* base = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  const uint32_t ring_s = smem_u32(base);
  const uint32_t zero_s = ring_s + kLZeroOff;
  const uint32_t full_s = ring_s + kLBarOff;
  const uint32_t empty_s = full_s + kLRing * 8;
  float* const part = reinterpret_cast<float*>(base + kLPartOff);
  // per slot: unit, first chunk of the group, the block's unit sequence number,
  // chunks of the unit (ordered by the slot's mbarrier, whose arrival releases
  // and whose wait acquires)
  int4* const meta = reinterpret_cast<int4*>(base + kLMetaOff);
  int* const u_arrive = reinterpret_cast<int*>(base + kLUnitOff);           // [kLUnitSlots]
  volatile int* u_done = reinterpret_cast<volatile int*>(base + kLUnitOff) + kLUnitSlots;
  volatile int* s_flags = reinterpret_cast<volatile int*>(base + kLFlagOff);  // [0] gave up, [1] last block
  uint32_t* const s_ready = reinterpret_cast<uint32_t*>(base + kLReadyOff);   // producer only
  int* const s_dtab = reinterpret_cast<int*>(base + kLDtabOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kLZero / 4) reinterpret_cast<uint32_t*>(base + kLZeroOff)[threadIdx.x] = 0u;
  if (threadIdx.x < kLUnitSlots) {
    u_arrive[threadIdx.x] = 0;
    u_done[threadIdx.x] = threadIdx.x - kLUnitSlots;   // unit slot u is free for unit sequence u
  }
  if (threadIdx.x < kDtabMax / 32) s_ready[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLRing; ++s) {
      mbar_init(full_s + 8 * s, 1);
      mbar_init(empty_s + 8 * s, kLConsumers);
    }
    s_flags[0] = 0;
    s_flags[1] = 0;
#define QMOE_PREFETCH_MAP(M) \
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&M)) : "memory")
    QMOE_PREFETCH_MAP(tq1);
    QMOE_PREFETCH_MAP(ts1);
    QMOE_PREFETCH_MAP(tq2);
    QMOE_PREFETCH_MAP(ts2);
    QMOE_PREFETCH_MAP(tx);
    QMOE_PREFETCH_MAP(th);
#undef QMOE_PREFETCH_MAP
  }
  mbar_init_fence();
  __syncthreads();
  // routing, the decode table, x16 and the zeroed synchronisation words come
  // from the routing kernel
  pdl_wait();
  pdl_trigger();

  int* const claim = ws.dsync;
  int* const done_blocks = ws.dsync + 1;
  int* const fc1_done = ws.dsync + kSyncHeader;
  int* const arrivals = ws.dsync + kSyncHeader + kDtabMax;
  const int entries = ws.counters[3];
  // the producer's first claim is in flight while the block copies the decode table
  int first_unit = 0;
  if (warp == kLConsumers && lane == 0) first_unit = atomicAdd(claim, 1);
  for (int i = threadIdx.x * 4; i < entries * kDtabInts; i += blockDim.x * 4)
    *reinterpret_cast<int4*>(s_dtab + i) = __ldg(reinterpret_cast<const int4*>(ws.dtab + i));
  __syncthreads();

  const int N1 = 2 * p.I, N2 = p.H;
  const int rg1 = N1 / kLRows, rg2 = N2 / kLRows;
  const int n1 = entries * rg1, nunits = n1 + entries * rg2;
  const int nst1 = p.H / kLChunk, nst2 = p.I / kLChunk;
  const int qh = p.H / 32;                       // 32-row groups of an output row

  if (warp == kLConsumers) {
    // ---------------- producer: one elected lane
    if (lane == 0) {
      int slot = 0, issued = 0, useq = 0;
      uint32_t ph = 0;
      bool ok = true;
      int u = first_unit;
      while (ok && u < nunits) {
        const int next = atomicAdd(claim, 1);          // its latency hides behind this unit's copies
        const bool f1 = u < n1;
        const int uu = f1 ? u : u - n1;
        const int rgs = f1 ? rg1 : rg2;
        const int ei = uu / rgs, rg = uu - ei * rgs;
        const int* d = s_dtab + ei * kDtabInts;
        const int row0 = d[0] * (f1 ? N1 : N2) + rg * kLRows;
        const int cnt = d[2];
        const int a0 = f1 ? d[4] : d[1], a1 = f1 ? d[5] : d[1] + 1;
        const int nst = f1 ? nst1 : nst2;
        for (int j0 = 0; j0 < nst; j0 += kLGroup) {
          if (!mbar_wait_for(empty_s + 8 * slot, ph ^ 1u, kLWaitNs)) { ok = false; break; }
          const uint32_t sb = ring_s + slot * kLSlot, bar = full_s + 8 * slot;
          meta[slot] = make_int4(u, j0, useq, nst);
          // every box lands whole (chunks past the unit's end read as zeros)
          mbar_expect_tx(bar, kLCodes + kLRows * kLGroup * 16 + kLGroup * 512 * cnt);
          tma_load_3d(sb, f1 ? &tq1 : &tq2, bar, 0, j0, row0);
          tma_load_3d(sb + kLScale, f1 ? &ts1 : &ts2, bar, 0, j0, row0);
          if (!f1 && !((s_ready[ei >> 5] >> (ei & 31)) & 1u)) {
            // the activations are the entry's SwiGLU outputs: every fc1 unit of
            // the entry has stored its h16 values (once seen, for the rest of the call)
            if (ld_acquire(fc1_done + ei) < rg1) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire(fc1_done + ei) < rg1) {
                if (globaltimer_ns() - t0 > kLWaitNs) { ok = false; break; }
                __nanosleep(64);
              }
            }
            fence_proxy_async_global();
            s_ready[ei >> 5] |= 1u << (ei & 31);
          }
          // on a failed wait the copies still complete the slot (the data is not used)
          tma_load_2d(sb + kLAct, f1 ? &tx : &th, bar, 0, a0 * nst + j0);
          if (cnt > 1) tma_load_2d(sb + kLAct + kLGroup * 512, f1 ? &tx : &th, bar, 0, a1 * nst + j0);
          ++issued;
          if (++slot == kLRing) { slot = 0; ph ^= 1u; }
          if (!ok) break;
        }
        ++useq;
        u = next;
      }
      // end of work: a slot without copies tells the consumers to stop (it is not handed back)
      if (ok) {
        if (mbar_wait_for(empty_s + 8 * slot, ph ^ 1u, kLWaitNs)) {
          meta[slot] = make_int4(-1, 0, 0, 0);
          mbar_arrive(full_s + 8 * slot);
        } else {
          ok = false;
        }
      }
      if (!ok) {
        atomicExch(ws.counters + 2, kErrLayerTimeout);
        s_flags[0] = 1;
        // let this block's copies in flight land before its shared memory is released
        const int first = issued > kLRing ? issued - kLRing : 0;
        for (int j = first; j < issued; ++j)
          mbar_wait_for(full_s + 8 * (j % kLRing), (uint32_t)(j / kLRing) & 1u, kLDrainNs);
      }
    }
  } else {
    // ---------------- consumers: warp w multiplies chunk w of every slot
    const int w = warp;
    const int g = lane >> 2, c = lane & 3;
    const bool owner = (g & 3) == c;             // supplies the activations of MMA column g
    const int on = g >> 2;                       // that column's route within the entry
    const int n = c >> 1;                        // route of this lane's D columns
    // this lane's 16-byte code pieces of row g of chunk w: logical piece c (first
    // 128 K) and c + 4 (second), swizzled by (4 g + w) mod 8
    const uint32_t code_off = (uint32_t)g * (kLGroup * 128) + (uint32_t)w * 128 +
                              ((uint32_t)(c ^ ((4 * g + w) & 7)) << 4);
    const uint32_t scale_off = kLScale + (uint32_t)g * (kLGroup * 16) + (uint32_t)w * 16 + 4u * (c & 1);
    const uint32_t act_off = (uint32_t)(kLAct + on * (kLGroup * 512) + w * 512 + 64 * c);

    const __half2 ne_d = __float2half2_rn(-(1024.0f + 8.0f)), no_d = __float2half2_rn(-(1024.0f + 128.0f));
    const uint32_t ne_def = *reinterpret_cast<const uint32_t*>(&ne_d);
    const uint32_t no_def = *reinterpret_cast<const uint32_t*>(&no_d);
    constexpr uint32_t kMagic = 0x64006400u;

    float acc[2][4];
    bool f1 = true;
    int ei = 0, rg = 0, cnt = 0, pos0 = 0, ex = 0, e_rid = 0;
    float e_scale = 1.0f, e_w = 0.0f;
    int slot = 0;
    uint32_t ph = 0;
    for (;;) {
      if (!consumer_wait(full_s + 8 * slot, ph, s_flags)) {
        if (lane == 0) atomicExch(ws.counters + 2, kErrLayerTimeout);
        break;
      }
      const int4 m = meta[slot];
      if (m.x < 0) break;
      const int u = m.x, j = m.y + w, useq = m.z, nst = m.w;
      const uint32_t sb = ring_s + slot * kLSlot;
      if (j >= nst) {
        // no chunk of this unit for this warp in the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_s + 8 * slot);
        if (++slot == kLRing) { slot = 0; ph ^= 1u; }
        continue;
      }
      if (j < kLConsumers) {
        // this warp's first chunk of the unit: its operands for the epilogue
        f1 = u < n1;
        const int uu = f1 ? u : u - n1;
        const int rgs = f1 ? rg1 : rg2;
        ei = uu / rgs;
        rg = uu - ei * rgs;
        const int* d = s_dtab + ei * kDtabInts;
        ex = d[0];
        pos0 = d[1];
        cnt = d[2];
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
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          mma16816(tb[sub][0], ne_def, ne_def, no_def, no_def, bw[sub][4 * i], bw[sub][4 * i + 1]);
          mma16816(tb[sub][1], ne_def, ne_def, no_def, no_def, bw[sub][4 * i + 2], bw[sub][4 * i + 3]);
        }
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        // rows 16 rh + g and 16 rh + 8 + g: the swizzle term (4 row + w) mod 8 is
        // the same for both, so the second is 8 row pitches further
        const uint32_t cb = sb + code_off + rh * (16 * kLGroup * 128);
        const uint32_t sr = sb + scale_off + rh * (16 * kLGroup * 16);
        uint4 cw[2][2];
        uint32_t sw[2][2];
        // piece c + 4 sits 64 bytes away from piece c in the other half of the row
        const uint32_t cb1 = cb ^ 64u;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(cw[0][0].x), "=r"(cw[0][0].y), "=r"(cw[0][0].z), "=r"(cw[0][0].w) : "r"(cb));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+4096];\n"
                     : "=r"(cw[0][1].x), "=r"(cw[0][1].y), "=r"(cw[0][1].z), "=r"(cw[0][1].w) : "r"(cb));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(cw[1][0].x), "=r"(cw[1][0].y), "=r"(cw[1][0].z), "=r"(cw[1][0].w) : "r"(cb1));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+4096];\n"
                     : "=r"(cw[1][1].x), "=r"(cw[1][1].y), "=r"(cw[1][1].z), "=r"(cw[1][1].w) : "r"(cb1));
        asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(sw[0][0]) : "r"(sr));
        asm volatile("ld.shared.u32 %0, [%1+512];\n" : "=r"(sw[0][1]) : "r"(sr));
        asm volatile("ld.shared.u32 %0, [%1+8];\n" : "=r"(sw[1][0]) : "r"(sr));
        asm volatile("ld.shared.u32 %0, [%1+520];\n" : "=r"(sw[1][1]) : "r"(sr));
        float t[2][2][4];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub)
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) t[sub][q][e] = 0.f;
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
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          float s_a0, s_a1, s_b0, s_b1;
          const uint32_t swa = sw[sub][0], swb = sw[sub][1];
          if constexpr (BF16S) {
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
      // every lane's shared-memory reads of the slot are done: hand it back
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_s + 8 * slot);
      if (++slot == kLRing) { slot = 0; ph ^= 1u; }
      if (j + kLConsumers < nst) continue;       // this warp has a later chunk of the unit

      // ---- this warp's last chunk of the unit: hand its sums over, the last warp finishes the unit
      const int npos = nst < kLConsumers ? nst : kLConsumers;
      const int us = useq % kLUnitSlots;
      float v[2][2];                             // [row half][row g, row g + 8], route n
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        v[rh][0] = acc[rh][0] + acc[rh][1];
        v[rh][1] = acc[rh][2] + acc[rh][3];
        v[rh][0] += __shfl_xor_sync(0xffffffffu, v[rh][0], 1);
        v[rh][1] += __shfl_xor_sync(0xffffffffu, v[rh][1], 1);
      }
      // the unit slot is free once the unit kLUnitSlots earlier has been finished
      if (!smem_wait_eq(u_done + us, useq - kLUnitSlots)) {
        if (lane == 0) atomicExch(ws.counters + 2, kErrLayerTimeout);
        break;
      }
      float* ps = part + (us * kLConsumers + w) * 64;   // warp w holds chunks w, w + 4, ...
      if ((c & 1) == 0) {
        ps[0 * 16 + (lane >> 1)] = v[0][0];
        ps[1 * 16 + (lane >> 1)] = v[0][1];
        ps[2 * 16 + (lane >> 1)] = v[1][0];
        ps[3 * 16 + (lane >> 1)] = v[1][1];
      }
      __syncwarp();
      int arrived = 0;
      if (lane == 0) {
        __threadfence_block();
        arrived = atomicAdd(u_arrive + us, 1);
      }
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (arrived != npos - 1) continue;
      // the unit's sums, warp positions in K order
      __syncwarp();
      __threadfence_block();
      const float* pb = part + us * kLConsumers * 64 + (lane >> 1);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float sum = pb[r * 16];
        for (int q = 1; q < npos; ++q) sum += pb[q * 64 + r * 16];
        v[r >> 1][r & 1] = sum;
      }
      __syncwarp();
      if (lane == 0) {
        u_arrive[us] = 0;
        __threadfence_block();
        u_done[us] = useq;                       // the slot's partial sums are read
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
            const float h_lo = silu(v[rh][0] * inv + b_lo.x) * (up_lo * inv + b_lo.y) * sigma * sigma;
            const float h_hi = silu(v[rh][1] * inv + b_hi.x) * (up_hi * inv + b_hi.y) * sigma * sigma;
            // fc2 reads these as activations: K-order permuted, odd K positions carry 1/16
            const int pj0 = (j_lo & ~7) + ((j_lo & 7) < 4 ? 2 * (j_lo & 7) : 2 * (j_lo & 7) - 7);
            const int pj1 = (j_hi & ~7) + ((j_hi & 7) < 4 ? 2 * (j_hi & 7) : 2 * (j_hi & 7) - 7);
            ws.h16[(int64_t)hp * p.I + pj0] = __half_as_ushort(__float2half_rn((j_lo & 1) ? h_lo * 0.0625f : h_lo));
            ws.h16[(int64_t)hp * p.I + pj1] = __half_as_ushort(__float2half_rn((j_hi & 1) ? h_hi * 0.0625f : h_hi));
          }
        }
        // publish: the unit's h16 values are stored (the release orders the
        // other lanes' stores, which the warp barrier ordered before it)
        __syncwarp();
        if (lane == 0) red_add_release(fc1_done + ei, 1);
      } else {
        const float inv = 1.0f / e_scale;
        const float fct = inv * inv * e_w;
        if ((c & 1) == 0 && n < cnt) {
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            const int row = rg * kLRows + 16 * rh + g;
            __stcg(ws.y + (int64_t)e_rid * p.H + row, v[rh][0] * fct);
            __stcg(ws.y + (int64_t)e_rid * p.H + row + 8, v[rh][1] * fct);
          }
        }
        // combine: count the unit's 32 rows of each of its routes' tokens; the
        // unit that brings a token's k-th route for these rows writes them out
        __syncwarp();
        const int rid0 = __shfl_sync(0xffffffffu, e_rid, 0), rid1 = __shfl_sync(0xffffffffu, e_rid, 2);
        int last = 0;
        if (lane < cnt) {
          const int tok = (lane ? rid1 : rid0) / p.k;
          last = atom_add_acq_rel(arrivals + (int64_t)tok * qh + rg, 1) == p.k - 1;
        }
        const uint32_t lastm = __ballot_sync(0xffffffffu, last);
        __syncwarp();
        for (int r = 0; r < 2; ++r) {
          if (!((lastm >> r) & 1u)) continue;
          const int64_t tok = (r ? rid1 : rid0) / p.k;
          const int row = rg * kLRows + lane;
          float sum = 0.0f;
          // routes in batches of 8: every load of a batch is issued before the first add
          for (int j0 = 0; j0 < p.k; j0 += 8) {
            float wj[8], yv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int64_t rr = tok * p.k + (j0 + q < p.k ? j0 + q : j0);
              wj[q] = j0 + q < p.k ? __ldg(ws.topk_w + rr) : 0.0f;
              yv[q] = __ldcg(ws.y + rr * p.H + row);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (wj[q] == 0.0f) continue;           // also the batch's padding past k
              if (p.b2) {
                const int e = __ldg(ws.topk_idx + tok * p.k + j0 + q);
                sum += yv[q] + wj[q] * half_bits_to_float(p.b2[(int64_t)e * p.H + row], p.dtype);
              } else {
                sum += yv[q];
              }
            }
          }
          a.out[tok * p.H + row] = float_to_half_bits(sum, p.dtype);
        }
      }
    }
  }

  // the last block to finish turns the whole output into NaN if any wait gave up
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_flags[1] = atomicAdd(done_blocks, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (s_flags[1]) {
    __threadfence();
    if (*reinterpret_cast<volatile int*>(ws.counters + 2) != 0) {
      const uint16_t nan = p.dtype == QMOE_BF16 ? 0x7FC0u : 0x7E00u;
      for (int64_t i = threadIdx.x; i < p.T * p.H; i += blockDim.x) a.out[i] = nan;
    }
  }
}

}  // namespace

bool decode_layer_applies(const Problem& p, bool has_zp) {
  return !has_zp && p.path == QMOE_PATH_DECODE && p.bits == 4 && p.block == 32 && p.T <= kDecodeMaxT &&
         p.H % kLChunk == 0 && p.I % kLChunk == 0;
}

cudaError_t launch_decode_layer(const Problem& p, const uint8_t* fc1_q, const void* fc1_scales,
                                const uint8_t* fc2_q, const void* fc2_scales, const Workspace& ws,
                                void* out, cudaStream_t s) {
  const uint64_t rows1 = (uint64_t)p.E * 2 * p.I, rows2 = (uint64_t)p.E * p.H;
  const uint64_t nst1 = (uint64_t)p.H / kLChunk, nst2 = (uint64_t)p.I / kLChunk;
  // codes and scales as [rows][chunk][piece] (pieces of 128 B of codes, 8 scales);
  // activations as [row * chunks + chunk][256]
  CUtensorMap tq1, ts1, tq2, ts2, tx, th;
  if (!make_map_3d(&tq1, CU_TENSOR_MAP_DATA_TYPE_UINT8, fc1_q, 128, nst1, rows1, 128, (uint64_t)p.H / 2, 128,
                   kLGroup, kLRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&ts1, CU_TENSOR_MAP_DATA_TYPE_UINT16, fc1_scales, 8, nst1, rows1, 16, (uint64_t)p.H / 16, 8,
                   kLGroup, kLRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_3d(&tq2, CU_TENSOR_MAP_DATA_TYPE_UINT8, fc2_q, 128, nst2, rows2, 128, (uint64_t)p.I / 2, 128,
                   kLGroup, kLRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&ts2, CU_TENSOR_MAP_DATA_TYPE_UINT16, fc2_scales, 8, nst2, rows2, 16, (uint64_t)p.I / 16, 8,
                   kLGroup, kLRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT16, ws.x16, kLChunk, (uint64_t)p.T * nst1, kLChunk * 2,
                   kLChunk, kLGroup, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT16, ws.h16, kLChunk, (uint64_t)p.R() * nst2, kLChunk * 2,
                   kLChunk, kLGroup, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  LayerArgs a{p, ws, static_cast<uint16_t*>(out)};
  // the decode table's share of shared memory is sized by the entries it can hold
  int64_t entries = (int64_t)p.E * ((p.T + 1) / 2);
  if (entries > p.R()) entries = p.R();
  const size_t smem = (size_t)kLSmemFixed + (size_t)entries * kDtabInts * 4;
  const int per_sm = 3 * (smem + 1024) <= 228 * 1024 ? 3 : 2;
  const int blocks = device_sm_count() * per_sm;
  if (p.dtype == QMOE_BF16) {
    const cudaError_t err = ensure_smem_optin(decode_layer_kernel<true>, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(decode_layer_kernel<true>, dim3(blocks), dim3(kLThreads), smem, s, tq1, ts1, tq2, ts2,
                      tx, th, a);
  }
  const cudaError_t err = ensure_smem_optin(decode_layer_kernel<false>, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(decode_layer_kernel<false>, dim3(blocks), dim3(kLThreads), smem, s, tq1, ts1, tq2, ts2,
                    tx, th, a);
}

}  // namespace qmoe
