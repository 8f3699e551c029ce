// qmoe_internal.cuh -- shared declarations of the QMoE CUDA path (sm_103a).
//
// Layout of the caller's workspace, launcher declarations and small device
// helpers used by more than one kernel file.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/qmoe.h"

namespace qmoe {

constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
constexpr int kPermuteChunk = 512;    // routes per block in the grouping kernels
// The decode path (expert weights streamed once, the routes of an expert on the
// MMA's N side) takes batches of up to 64 tokens and kPermuteChunk routes: the
// one-block routing kernel groups them and builds the decode table. AUTO picks
// it for T <= 8 and, above that, while the routes number fewer than 4 per
// expert (below 64 routes in all, always): the pages switch from their
// tensor-core GEMV to the grouped GEMM at num_r >= 64 && num_r >= 4 E.
// Wall-time limit of every bounded wait in the matmul kernels (1 s: far beyond
// any legitimate wait). A test build sets it to 0, so that waits run out and
// the kernels' give-up paths run (tests/test_gpu_wait_timeouts.py).
#ifndef QMOE_WAIT_LIMIT_NS
#define QMOE_WAIT_LIMIT_NS 1000000000ull
#endif

constexpr int kDecodeMaxT = 64;
constexpr int kDecodeChunk = 8;       // routes of one expert per MMA N-fragment (generic decode kernel)
constexpr int kTileM = 256;           // rows (routes) per grouped-GEMM tile
constexpr int kTileWs = 128;          // rows per tile of the weights-stationary grouped GEMM
constexpr int kDtabInts = 8;          // ints per decode-table entry
constexpr int kDtabMax = kPermuteChunk;  // entries: at most one per route

// ---------------------------------------------------------------------------
// Workspace: every scratch buffer of one forward call, carved from the
// caller's allocation at 256-byte aligned offsets.
// ---------------------------------------------------------------------------
struct Workspace {
  int32_t* topk_idx;      // [R]      expert of route r = t*k + j
  float* topk_w;          // [R]      routing weight of route r
  float* tok_scale;       // [T]      power of two that brings max|x_t| into [1, 2)
  uint16_t* x16;          // [T][H]   FP16 bits of x_t * tok_scale[t], K-order permuted
  int32_t* offsets;       // [E+1]    exclusive prefix of per-expert route counts
  int32_t* sorted_route;  // [R]      route ids grouped by expert, stable
  int32_t* active;        // [E + R/8] experts with at least one route, ascending; on the
                          //   decode path one word per (expert, chunk of up to 8 of its
                          //   routes): expert | chunk << 16
  int32_t* counters;      // [4]      [0] active experts (decode path: chunks), [1] grouped
                          //   tiles, [2] error flag,
                          //          [3] decode-table entries
  int32_t* tiles;         // [2*max_tiles] (expert, first sorted row) of each tile (Problem::tile_m rows)
  int32_t* chunk_hist;    // [nchunks][E] per-chunk expert counts, then chunk bases
  int32_t* dtab;          // [kDtabMax][kDtabInts] decode table: one entry per (active expert,
                          //   pair of its routes): expert, first sorted row of the pair, routes in
                          //   the pair (1 or 2), route id of the first, token of each route, route
                          //   id of the second (0 if none), the expert's h_norm (FP32 bits);
                          //   counters[3] entries
  uint16_t* x16s;         // [R][H]   x16 rows gathered into sorted-route order (grouped)
  uint16_t* h16;          // [R][I]   SwiGLU output, FP16, sorted-route order, K-order permuted
  float* y;               // [R][H]   weighted fc2 output per route id (FP32)
  uint16_t* rlogits;      // [T][E]   router logits computed from x (qmoe_options.router_weight)
  float* dsplit;           // decode split-K partials [work items][4][32] (FP32)
  int32_t* dticket;        // [decode units] arrival counters of the split-K partials
  int32_t* dsync;          // decode layer kernel: [0] unit claims, [kSyncHeader ..] fc1
                           //   completions per decode-table entry [kDtabMax]; zeroed by the
                           //   routing kernel of every decode-path call
  int64_t dsync_ints;      // capacity of dsync
  int64_t dunits_max;      // capacity of dticket
  int64_t dsplit_items;    // capacity of dsplit in work items
  int64_t max_tiles;
  int64_t nchunks;
};

struct Problem {
  int64_t T;
  int H, I, E, k, bits, block, dtype, path;
  int full_softmax;               // routing weights under the softmax over all E logits
  const uint16_t* b1;             // [E][2I] fc1 bias in dtype, or null
  const uint16_t* b2;             // [E][H]  fc2 bias in dtype, or null
  const uint16_t* s1;             // fc1 block scales [E][2I][H/block] in dtype (read by h_norm)
  const uint8_t* s1b;             // the same for the FP4 formats (8-bit scales)
  int format;                     // qmoe_format of the expert weights
  const float* g1;                // NVFP4: per-expert FP32 global scales of fc1 / fc2, or null
  const float* g2;
  int logits_after_wait;          // the router logits are the previous kernel's output: read
                                  //   them only after pdl_wait()
  int tile_m;                     // grouped path: sorted rows per tile, kTileM (route tiles) or
                                  //   kTileWs (weights-stationary kernel; grouped_ws)
  __host__ __device__ int64_t R() const { return T * (int64_t)k; }
};

// The path a problem runs on (QMOE_PATH_DECODE or QMOE_PATH_GROUPED; AUTO resolved).
int resolve_path(const qmoe_problem& p);

// Whether the grouped path runs the weights-stationary kernel (an expert's
// routes on the MMA N side) rather than route tiles: when the routes per expert
// are few on average (R <= kWsRoutesPerExpert * E), or as `force` asks
// (0 automatic, 1 route tiles, 2 weights-stationary: QMOE_PATH_GROUPED_ROUTE_TILES
// and QMOE_PATH_GROUPED_WS). It reads codes in copies of kWsCodeK along K, so
// hidden and inter must be multiples of kWsCodeK.
constexpr int kWsRoutesPerExpert = 32;
constexpr int kWsCodeK = 256;
__host__ __device__ inline bool grouped_ws_applies(int H, int I) { return H % kWsCodeK == 0 && I % kWsCodeK == 0; }
__host__ __device__ inline bool grouped_ws(int64_t R, int E, int H, int I, int force) {
  if (force == 1 || !grouped_ws_applies(H, I)) return false;
  if (force == 2) return true;
  return R <= (int64_t)kWsRoutesPerExpert * E;
}

// Decode work units (decode-table entries x 16-row groups of the larger matmul)
// and split-K work items the workspace is sized for.
int64_t decode_units_max(const Problem& p);
int64_t decode_split_items_max(const Problem& p);

// Synchronisation words of the decode-layer kernel (see Workspace::dsync).
constexpr int kSyncHeader = 4;
__host__ __device__ inline int64_t decode_sync_ints(const Problem&) { return kSyncHeader + kDtabMax; }

// Byte size of the workspace for problem p and the pointers inside `base`
// (base may be null when only the size is wanted).
size_t workspace_layout(const Problem& p, bool grouped, void* base, Workspace* ws);

// K-order permutation group: positions 2i and 2i+1 of each group hold elements
// i and i + G/2. G = 8 for 4-bit codes and 16 for 2- and 3-bit codes. It lets
// the dequantisers produce FP16 pairs straight from the packed words.
__host__ __device__ inline int perm_group(int bits) { return bits == 4 ? 8 : 16; }

// The INT4 decode kernel with per-block scales applied after the MMA (block 32,
// K a multiple of 128 for both matmuls). It reads activations whose odd K
// positions are pre-divided by 16 (see decode.cu).
__host__ __device__ inline bool decode_int4_blockscaled(const Problem& p) {
  return p.path == QMOE_PATH_DECODE && p.format == QMOE_FORMAT_INT && p.bits == 4 && p.block == 32 &&
         p.H % 128 == 0 && p.I % 128 == 0;
}

// How the routing kernel writes x16: not at all, plain, or with the odd K
// positions divided by 16 (for decode_int4_blockscaled).
// kX16Natural: plain values in natural K order (the decode layer kernel's FP4
// path, whose operand pairs are adjacent codes).
enum X16Mode { kX16None = 0, kX16Plain = 1, kX16OddSixteenth = 2, kX16Natural = 3 };

// ---------------------------------------------------------------------------
// launchers (return the launch error, never synchronise)
// ---------------------------------------------------------------------------
cudaError_t launch_route(const Problem& p, const void* x, const void* logits, const Workspace& ws,
                         int x16_mode, cudaStream_t s);
cudaError_t launch_group(const Problem& p, const Workspace& ws, bool want_tiles, cudaStream_t s);
cudaError_t launch_gather(const Problem& p, const Workspace& ws, cudaStream_t s);
// One expert matmul stage: fc1 (with SwiGLU) when fc1 is true, else fc2.
cudaError_t launch_decode(const Problem& p, bool fc1, const uint8_t* q, const void* scales,
                          const uint8_t* zp, const Workspace& ws, cudaStream_t s);
cudaError_t launch_grouped(const Problem& p, bool fc1, const uint8_t* q, const void* scales,
                           const uint8_t* zp, const Workspace& ws, cudaStream_t s);
cudaError_t launch_combine(const Problem& p, const Workspace& ws, void* out, cudaStream_t s);
// Router logits [T][E] = x [T][H] . w_router [E][H]^T, rounded once to the dtype (router.cu).
cudaError_t launch_router_logits(const Problem& p, const void* x, const void* w_router, void* logits,
                                 cudaStream_t s);
// The decode layer's two expert matmuls (fc1 + SwiGLU, fc2) as one persistent
// kernel (decode_layer.cu); applies to INT4 block 32 without zero points, H and
// inter multiples of 256.
bool decode_layer_applies(const Problem& p, bool has_zp);
cudaError_t launch_decode_layer(const Problem& p, const uint8_t* fc1_q, const void* fc1_scales,
                                const uint8_t* fc2_q, const void* fc2_scales, const Workspace& ws,
                                cudaStream_t s);

// Per-device launch facts (launch_cache.cu), keyed by device and context and
// safe to call from several host threads.
int device_sm_count();
// The calling thread's device ordinal and current context (null before the
// runtime has made one current); false when no device is available.
bool current_device_context(int* dev, const void** ctx);
// Opt kernel fn into `bytes` of dynamic shared memory on the current device.
cudaError_t ensure_smem_optin(const void* fn, int bytes);
template <typename F>
cudaError_t ensure_smem_optin(F* fn, int bytes) {
  return ensure_smem_optin(reinterpret_cast<const void*>(fn), bytes);
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float half_bits_to_float(uint16_t b, int dtype) {
  if (dtype == QMOE_BF16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

// fc1 bias of SwiGLU unit j of expert e: gate (row 2j) and up (row 2j+1), or
// zeros without a bias.
__device__ __forceinline__ float2 fc1_bias_pair(const Problem& p, int e, int j) {
  if (!p.b1) return make_float2(0.0f, 0.0f);
  const uint32_t v = __ldg(reinterpret_cast<const unsigned int*>(p.b1 + ((int64_t)e * p.I + j) * 2));
  return make_float2(half_bits_to_float((uint16_t)(v & 0xFFFFu), p.dtype),
                     half_bits_to_float((uint16_t)(v >> 16), p.dtype));
}

// The SwiGLU output h is stored in FP16 as h * sigma_t^2 * rho_e (sigma_t: the
// token's activation scale) and the fc2 epilogue divides by the same product.
// h grows with the square of the fc1 weights, so rho_e is the power of two
// 2^(-2 (E + 7)) with 2^E <= |s| < 2^(E+1) for the expert's first fc1 block
// scale s (FP4 formats: its E8M0 value, or its E4M3 value times the expert's
// NVFP4 global scale): the stored values keep the magnitude that block scales near 2^-7
// give, whatever the scale range of the model (BF16 scales from 2^-40 to 2^40
// keep the FP16 intermediate inside its normal range as long as an expert's
// scales stay within about 2^6 of its first one). A zero, subnormal, infinite
// or NaN first scale gives rho_e = 1. With an fc1 bias, h also holds the
// bias's own contribution, so rho_e is capped at 1 there. rho_e is a power of
// two: the scaling is exact.
__device__ __forceinline__ float h_norm(const Problem& p, int e) {
  float s;
  const int64_t first = (int64_t)e * (2 * p.I) * (p.H / p.block);
  if (p.format == QMOE_FORMAT_INT) {
    if (!p.s1) return 1.0f;
    s = fabsf(half_bits_to_float(__ldg(p.s1 + first), p.dtype));
  } else {
    // FP4 formats: the E8M0 scale, or the E4M3 scale times the expert's global scale
    if (!p.s1b) return 1.0f;
    const uint32_t b = __ldg(p.s1b + first);
    if (p.format == QMOE_FORMAT_MXFP4) {
      if (b == 0xFFu) return 1.0f;
      s = ldexpf(1.0f, (int)b - 127);
    } else {
      s = fabsf(__half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3))));
      if (p.g1) s *= fabsf(__ldg(p.g1 + e));
    }
  }
  if (!(s >= 1.17549435e-38f) || s > 3.0e38f) return 1.0f;  // zero, subnormal, inf, NaN
  int ex = (int)((__float_as_uint(s) >> 23) & 0xFF) - 127;   // floor(log2 s)
  ex = min(max(ex, -40), 40);
  const float rho = ldexpf(1.0f, -2 * (ex + 7));
  return p.b1 ? fminf(rho, 1.0f) : rho;
}

// Round to nearest even; NaN stays NaN (the CUDA conversion intrinsics).
__device__ __forceinline__ uint16_t float_to_half_bits(float v, int dtype) {
  if (dtype == QMOE_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

// Programmatic dependent launch. Every kernel of the path is launched so that it
// may be scheduled while the previous kernel on the stream is still running.
// pdl_wait() returns once the previous kernel has completed and its writes are
// visible; a kernel touches nothing that kernel writes, nor memory that it
// reads, before pdl_wait(). pdl_trigger() lets the next kernel be scheduled
// (once every block of this one has called it or exited); a kernel calls it
// only after pdl_wait(), except the fc2 and combine kernels, whose dependents
// wait for them before touching anything. The results do not change.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// D += A B on the legacy tensor path: m16n8k16, FP16 operands, FP32 accumulators.
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a & mask) | orv in one LOP3.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
  return d;
}

}  // namespace qmoe
