// route.cu -- per-token top-k routing and token->expert grouping (sm_103a).
//
// route_topk_softmax: one warp per token. The k largest raw router logits are
// selected by k rounds of a warp-wide maximum over (order key, expert) pairs,
// so ties go to the lower expert index, and the weights are the softmax over
// the selected logits ("Document and test packed token inputs for MoE and
// QMoE" #32522: QMoE receives raw logits; the kernel applies top-k and then
// normalises, the reference being a softmax over the top-k logits). Warps also
// convert each token's activations to the FP16 operand of the matmuls. For a
// small batch (at most 512 routes) one block does routing and grouping from the
// logits alone, in shared memory, while the previous kernel on the stream may
// still run, and writes the results and converts the activations after it.
//
// expert_histogram_scan_permute: a stable counting sort of the T*k route ids by
// expert (the sorted expert map / expert_first_token_offset that the pages'
// grouped kernels consume, "[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload
// ..." #33731 items 1-2). Per-chunk histograms, one scan, and a scatter that
// ranks equal experts by route id with warp match masks, so the result is the
// unique stable order, bit for bit, whatever the scheduling.
#include "qmoe_internal.cuh"

namespace qmoe {
namespace {

constexpr int kGroupThreads = 512;
static_assert(kPermuteChunk % kGroupThreads == 0, "chunk must be a multiple of the block");

// Order key of a logit: larger logit -> larger key; +0 and -0 equal; NaN lowest.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;
  if (v == 0.0f) return 0x80000000u;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ void convert_token(const Problem& p, const uint16_t* __restrict__ x, const Workspace& ws,
                              int64_t t, int x16_mode);

// Top-k + softmax of token t (whole warp), and optionally its FP16 activations.
template <int PER_LANE>
__device__ void route_token(const Problem& p, const uint16_t* __restrict__ x,
                            const uint16_t* __restrict__ logits, const Workspace& ws, int64_t t,
                            int x16_mode, int* s_idx = nullptr, float* s_w = nullptr) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, k = p.k;
  const uint16_t* lrow = logits + t * E;
  uint64_t cand[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    cand[i] = 0;
    if (e < E) {
      const float v = half_bits_to_float(lrow[e], p.dtype);
      cand[i] = ((uint64_t)order_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
    }
  }
  int my_e = 0;
  float my_l = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) best = cand[i] > best ? cand[i] : best;
    best = warp_max_u64(best);
    const int e = (int)(0xFFFFFFFFu - (uint32_t)best);
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i)
      if (lane + 32 * i == e) cand[i] = 0;
    if (lane == j) {
      my_e = e;
      my_l = half_bits_to_float(lrow[e], p.dtype);
    }
  }
  // softmax over the selected logits, shifted by the largest (j = 0); with
  // full_softmax the denominator runs over all E logits of the token
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  float denom = 0.0f;
  if (p.full_softmax) {
    for (int e = lane; e < E; e += 32) denom += expf(half_bits_to_float(lrow[e], p.dtype) - l0);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  } else {
    for (int j = 0; j < k; ++j) denom += expf(__shfl_sync(0xffffffffu, my_l, j) - l0);
  }
  if (lane < k) {
    const float w = expf(my_l - l0) / denom;
    if (s_w) {                                   // shared memory only; written out later
      s_idx[t * k + lane] = my_e;
      s_w[t * k + lane] = w;
    } else {
      ws.topk_idx[t * k + lane] = my_e;
      ws.topk_w[t * k + lane] = w;
      if (s_idx) s_idx[t * k + lane] = my_e;
    }
  }
  if (x16_mode == kX16None) return;
  convert_token(p, x, ws, t, x16_mode);
}

// Activations of token t (whole warp): scale by a power of two so that max|x_t|
// lies in [1, 2), round to FP16, and store in the K-order permutation of the
// dequantisers.
__device__ void convert_token(const Problem& p, const uint16_t* __restrict__ x, const Workspace& ws,
                              int64_t t, int x16_mode) {
  const int lane = threadIdx.x & 31;
  const int H = p.H;
  const uint16_t* xrow = x + t * (int64_t)H;
  float m = 0.0f;
  for (int base = lane * 16; base < H; base += 32 * 16) {
    const uint4 a = *reinterpret_cast<const uint4*>(xrow + base);
    const uint4 b = *reinterpret_cast<const uint4*>(xrow + base + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      m = fmaxf(m, fabsf(half_bits_to_float((uint16_t)(w[i] & 0xFFFF), p.dtype)));
      m = fmaxf(m, fabsf(half_bits_to_float((uint16_t)(w[i] >> 16), p.dtype)));
    }
  }
  m = warp_max_f(m);
  float sigma = 1.0f;
  if (m > 0.0f && m <= 3.4e38f) {
    int ex;
    frexpf(m, &ex);                   // m = f * 2^ex, f in [0.5, 1)
    int sh = 1 - ex;                  // m * 2^sh in [1, 2)
    sh = sh > 60 ? 60 : (sh < -60 ? -60 : sh);
    sigma = ldexpf(1.0f, sh);
  }
  if (lane == 0) ws.tok_scale[t] = sigma;
  const int G = perm_group(p.bits);
  uint16_t* orow = ws.x16 + t * (int64_t)H;
  for (int base = lane * 16; base < H; base += 32 * 16) {
    const uint4 a = *reinterpret_cast<const uint4*>(xrow + base);
    const uint4 b = *reinterpret_cast<const uint4*>(xrow + base + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint16_t in[16], out[16];
    // odd K positions carry 1/16 in the block-scaled INT4 decode layout
    const float odd = x16_mode == kX16OddSixteenth ? sigma * 0.0625f : sigma;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      in[2 * i] = __half_as_ushort(__float2half_rn(half_bits_to_float((uint16_t)(w[i] & 0xFFFF), p.dtype) * sigma));
      in[2 * i + 1] = __half_as_ushort(__float2half_rn(half_bits_to_float((uint16_t)(w[i] >> 16), p.dtype) * odd));
    }
    if (x16_mode == kX16Natural) {
#pragma unroll
      for (int i = 0; i < 16; ++i) out[i] = in[i];
    } else if (G == 8) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          out[8 * g + 2 * i] = in[8 * g + i];
          out[8 * g + 2 * i + 1] = in[8 * g + i + 4];
        }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        out[2 * i] = in[i];
        out[2 * i + 1] = in[i + 8];
      }
    }
    uint4 o0, o1;
    o0.x = out[0] | ((uint32_t)out[1] << 16);
    o0.y = out[2] | ((uint32_t)out[3] << 16);
    o0.z = out[4] | ((uint32_t)out[5] << 16);
    o0.w = out[6] | ((uint32_t)out[7] << 16);
    o1.x = out[8] | ((uint32_t)out[9] << 16);
    o1.y = out[10] | ((uint32_t)out[11] << 16);
    o1.z = out[12] | ((uint32_t)out[13] << 16);
    o1.w = out[14] | ((uint32_t)out[15] << 16);
    *reinterpret_cast<uint4*>(orow + base) = o0;
    *reinterpret_cast<uint4*>(orow + base + 8) = o1;
  }
}

template <int PER_LANE>
__global__ void __launch_bounds__(256) route_kernel(Problem p, const uint16_t* __restrict__ x,
                                                    const uint16_t* __restrict__ logits,
                                                    Workspace ws, int x16_mode) {
  pdl_wait();
  pdl_trigger();
  const int warps = blockDim.x >> 5;
  for (int64_t t = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); t < p.T;
       t += (int64_t)gridDim.x * warps)
    route_token<PER_LANE>(p, x, logits, ws, t, x16_mode);
}

// ---------------------------------------------------------------------------
// grouping
// ---------------------------------------------------------------------------

// Exclusive scan of one int per thread over the whole block (up to 1024 threads).
__device__ int block_exclusive_scan(int v, int* sh /* >= 32 ints */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    if (lane < nw) sh[lane] = s;  // inclusive per-warp totals
  }
  __syncthreads();
  const int warp_base = warp ? sh[warp - 1] : 0;
  const int result = warp_base + incl - v;
  if (total) *total = sh[(blockDim.x >> 5) - 1];
  __syncthreads();
  return result;
}

// Count of routes per expert in routes [r0, r1) into shared hist (pre-zeroed).
__device__ void count_routes(const int32_t* __restrict__ idx, int64_t r0, int64_t r1, int* hist) {
  for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) atomicAdd(&hist[idx[r]], 1);
}

// Stable scatter of routes [r0, r1): position = base[e] + (routes of e before r
// in this range). base is in shared memory and is advanced past the range.
// warp_cnt holds (blockDim/32) * E ints of shared scratch.
__device__ void scatter_routes(const int32_t* __restrict__ idx, int64_t r0, int64_t r1, int E,
                               int* base, int* warp_cnt, int32_t* __restrict__ sorted_route) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int64_t round0 = r0; round0 < r1; round0 += blockDim.x) {
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) warp_cnt[i] = 0;
    __syncthreads();
    const int64_t r = round0 + threadIdx.x;
    const bool valid = r < r1;
    const int e = valid ? idx[r] : -1 - lane;  // invalid lanes never match a real expert
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) warp_cnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += warp_cnt[w * E + e];
      sorted_route[base[e] + before + rank] = (int32_t)r;
    }
    __syncthreads();
    // advance the bases past this round
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
      int n = 0;
      for (int w = 0; w < nw; ++w) n += warp_cnt[w * E + ee];
      base[ee] += n;
    }
    __syncthreads();
  }
}

// Offsets, active-expert list and the tile list (tiles of tile_m sorted rows)
// from per-expert totals held one per thread (thread e < E holds total[e]).
__device__ void finish_groups(int E, int total_e, const Workspace& ws, bool want_tiles, int tile_m, int* sh,
                              int* expert_base_out) {
  const int e = threadIdx.x;
  const int v = e < E ? total_e : 0;
  int R_total;
  const int off = block_exclusive_scan(v, sh, &R_total);
  if (e < E) ws.offsets[e] = off;
  if (e == 0) ws.offsets[E] = R_total;
  if (expert_base_out && e < E) expert_base_out[e] = off;
  int n_active;
  const int apos = block_exclusive_scan(v > 0 ? 1 : 0, sh, &n_active);
  if (e < E && v > 0) ws.active[apos] = e;
  if (e == 0) {
    ws.counters[0] = n_active;
    ws.counters[2] = 0;  // error flag of the grouped GEMM (set on a timed-out wait)
  }
  if (want_tiles) {
    const int nt = (v + tile_m - 1) / tile_m;
    int n_tiles;
    const int tpos = block_exclusive_scan(nt, sh, &n_tiles);
    for (int i = 0; i < nt; ++i) {
      ws.tiles[2 * (tpos + i)] = e;
      ws.tiles[2 * (tpos + i) + 1] = off + i * tile_m;
    }
    if (e == 0) ws.counters[1] = n_tiles;
  }
}

__global__ void __launch_bounds__(kGroupThreads) group_count_kernel(Problem p, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  int* hist = smem;
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t R = p.R();
  const int64_t r0 = (int64_t)blockIdx.x * kPermuteChunk;
  const int64_t r1 = r0 + kPermuteChunk < R ? r0 + kPermuteChunk : R;
  count_routes(ws.topk_idx, r0, r1, hist);
  __syncthreads();
  for (int i = threadIdx.x; i < p.E; i += blockDim.x)
    ws.chunk_hist[(int64_t)blockIdx.x * p.E + i] = hist[i];
}

// Per-expert exclusive prefix of the per-chunk counts, plus the expert bases:
// thread (part, e) sums chunks [nc*part/P, nc*(part+1)/P) of expert e (P parts
// per expert, coalesced over e), the parts are scanned per expert, and a second
// pass writes every chunk's base. Loads go eight chunks at a time.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) group_scan_kernel(Problem p, Workspace ws, int want_tiles) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sh[32];
  __shared__ int part_sum[kScanThreads];
  __shared__ int expert_base[kMaxExperts];
  const int E = p.E;
  int P = 1;
  while (2 * P * E <= kScanThreads) P *= 2;
  const int tid = threadIdx.x;
  const bool active = tid < P * E;
  const int e = tid % E, part = tid / E;
  const int64_t nc = ws.nchunks;
  const int64_t c_lo = nc * part / P, c_hi = nc * (part + 1) / P;
  int32_t* __restrict__ h = ws.chunk_hist;
  int sum = 0;
  if (active)
    for (int64_t c0 = c_lo; c0 < c_hi; c0 += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = c0 + u < c_hi ? h[(c0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += v[u];
    }
  part_sum[tid] = active ? sum : 0;
  __syncthreads();
  int total = 0;
  if (tid < E)
    for (int q = 0; q < P; ++q) {
      const int v = part_sum[q * E + tid];
      part_sum[q * E + tid] = total;
      total += v;
    }
  __syncthreads();
  finish_groups(E, total, ws, want_tiles != 0, p.tile_m, sh, expert_base);
  __syncthreads();
  if (active) {
    int run = expert_base[e] + part_sum[tid];
    for (int64_t c0 = c_lo; c0 < c_hi; c0 += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = c0 + u < c_hi ? h[(c0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + u < c_hi) {
          h[(c0 + u) * E + e] = run;
          run += v[u];
        }
    }
  }
}

__global__ void __launch_bounds__(kGroupThreads) group_scatter_kernel(Problem p, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  int* base = smem;                 // [E]
  int* warp_cnt = smem + p.E;       // [16][E]
  for (int i = threadIdx.x; i < p.E; i += blockDim.x)
    base[i] = ws.chunk_hist[(int64_t)blockIdx.x * p.E + i];
  __syncthreads();
  const int64_t R = p.R();
  const int64_t r0 = (int64_t)blockIdx.x * kPermuteChunk;
  const int64_t r1 = r0 + kPermuteChunk < R ? r0 + kPermuteChunk : R;
  scatter_routes(ws.topk_idx, r0, r1, p.E, base, warp_cnt, ws.sorted_route);
}

// Routing and grouping of a small batch (R <= kPermuteChunk) in one block. All of
// it is computed in shared memory from the router logits alone, before the
// previous kernel on the stream has finished (programmatic dependent launch);
// then the kernel waits for it and writes the results, the decode table and the
// FP16 activations (which read x, the previous kernel's output).
// Dynamic shared memory: hist [E], warp_cnt [16][E], decode table [dtab_max][8].
template <int PER_LANE>
__global__ void __launch_bounds__(kGroupThreads) route_group_small_kernel(
    Problem p, const uint16_t* __restrict__ x, const uint16_t* __restrict__ logits, Workspace ws,
    int x16_mode, int want_tiles) {
  // logits computed by the previous kernel (the router GEMM) are read after its end
  if (p.logits_after_wait) pdl_wait();
  extern __shared__ int smem[];
  int* hist = smem;                  // [E]
  int* warp_cnt = smem + p.E;        // [16][E]
  int* s_dtab = warp_cnt + (kGroupThreads / 32) * p.E;   // [entries][kDtabInts] (decode path)
  __shared__ int sh[32];
  __shared__ int s_idx[kPermuteChunk];
  __shared__ float s_w[kPermuteChunk];
  __shared__ int s_sorted[kPermuteChunk];
  __shared__ int s_act[kMaxExperts + kPermuteChunk / kDecodeChunk];
  const int warps = blockDim.x >> 5;
  const int R = (int)p.R();
  const int e = threadIdx.x;
  for (int64_t t = threadIdx.x >> 5; t < p.T; t += warps)
    route_token<PER_LANE>(p, x, logits, ws, t, kX16None, s_idx, s_w);
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  count_routes(s_idx, 0, R, hist);
  __syncthreads();
  const int total = e < p.E ? hist[e] : 0;
  __syncthreads();
  int R_total, n_active, n_tiles = 0;
  const int off = block_exclusive_scan(total, sh, &R_total);
  // active list: on the decode path one word per (expert, chunk of up to
  // kDecodeChunk of its routes), expert | chunk << 16, so that the generic decode
  // kernel puts each chunk on one MMA N-fragment; otherwise one per expert
  const bool dec = p.path == QMOE_PATH_DECODE;  // (block-uniform) R <= kDtabMax on this path
  const int n_act_e = dec ? (total + kDecodeChunk - 1) / kDecodeChunk : (total > 0 ? 1 : 0);
  const int apos = block_exclusive_scan(n_act_e, sh, &n_active);
  const int nt = (total + p.tile_m - 1) / p.tile_m;
  const int tpos = want_tiles ? block_exclusive_scan(nt, sh, &n_tiles) : 0;
  if (e < p.E) {
    hist[e] = off;                   // scatter bases
    for (int i = 0; i < n_act_e; ++i) s_act[apos + i] = e | (i << 16);
  }
  __syncthreads();
  scatter_routes(s_idx, 0, R, p.E, hist, warp_cnt, s_sorted);   // ends with a block barrier
  // decode table: one entry per (active expert, pair of its routes), in expert
  // order, so that a decode work unit reaches its expert's rows and its tokens
  // with one independent load and always multiplies exactly one MMA column pair
  int n_entries = 0;
  if (dec) {
    const int first = block_exclusive_scan((total + 1) / 2, sh, &n_entries);
    for (int q = 0; 2 * q < total; ++q) {
      int* d = s_dtab + (first + q) * kDtabInts;
      const int cnt = total - 2 * q < 2 ? total - 2 * q : 2;
      d[0] = e;
      d[1] = off + 2 * q;
      d[2] = cnt;
      d[3] = s_sorted[off + 2 * q];
      d[4] = s_sorted[off + 2 * q] / p.k;
      d[5] = cnt > 1 ? s_sorted[off + 2 * q + 1] / p.k : 0;
      d[6] = cnt > 1 ? s_sorted[off + 2 * q + 1] : 0;
      d[7] = __float_as_int(h_norm(p, e));   // the expert's SwiGLU normalisation (fc1 scales are inputs)
    }
    __syncthreads();
  }

  // ---- the previous kernel has finished: write everything out
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    ws.topk_idx[i] = s_idx[i];
    ws.topk_w[i] = s_w[i];
    ws.sorted_route[i] = s_sorted[i];
  }
  if (e < p.E) ws.offsets[e] = off;
  if (e == 0) {
    ws.offsets[p.E] = R_total;
    ws.counters[0] = n_active;
    ws.counters[1] = n_tiles;
    ws.counters[2] = 0;  // error flag of the grouped GEMM / decode kernels (set on a timed-out wait)
    ws.counters[3] = n_entries;
  }
  for (int i = threadIdx.x; i < n_active; i += blockDim.x) ws.active[i] = s_act[i];
  if (want_tiles && e < p.E)
    for (int i = 0; i < nt; ++i) {
      ws.tiles[2 * (tpos + i)] = e;
      ws.tiles[2 * (tpos + i) + 1] = off + i * p.tile_m;
    }
  if (dec) {
    for (int64_t i = threadIdx.x; i < ws.dunits_max; i += blockDim.x) ws.dticket[i] = 0;
    for (int64_t i = threadIdx.x; i < ws.dsync_ints; i += blockDim.x) ws.dsync[i] = 0;
    for (int i = threadIdx.x; i < n_entries * kDtabInts; i += blockDim.x) ws.dtab[i] = s_dtab[i];
  }
  if (x16_mode != kX16None)
    for (int64_t t = threadIdx.x >> 5; t < p.T; t += warps) convert_token(p, x, ws, t, x16_mode);
}

__global__ void __launch_bounds__(256) gather_kernel(Problem p, Workspace ws) {
  pdl_wait();
  pdl_trigger();
  // x16s[pos] = x16[token of sorted route pos]; one warp per row, 16 bytes per
  // lane per access. Each lane issues all its loads of a 4-KB piece of the row
  // before its stores, so eight loads per lane are in flight at once.
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t R = p.R();
  const int chunks = p.H / 8;
  const uint16_t* __restrict__ x16 = ws.x16;
  uint16_t* __restrict__ x16s = ws.x16s;
  for (int64_t pos = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); pos < R;
       pos += (int64_t)gridDim.x * warps) {
    const int64_t t = ws.sorted_route[pos] / p.k;
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(x16 + t * p.H);
    uint4* __restrict__ dst = reinterpret_cast<uint4*>(x16s + pos * p.H);
    for (int c0 = 0; c0 < chunks; c0 += 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) v[u] = src[c];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) dst[c] = v[u];
      }
    }
  }
}

int num_sms() { return device_sm_count(); }

}  // namespace

cudaError_t launch_route(const Problem& p, const void* x, const void* logits, const Workspace& ws,
                         int x16_mode, cudaStream_t s) {
  const int64_t R = p.R();
  const bool small = R <= kPermuteChunk;
  const bool want_tiles = p.path == QMOE_PATH_GROUPED;
  const auto* xx = static_cast<const uint16_t*>(x);
  const auto* lg = static_cast<const uint16_t*>(logits);
  if (small) {
    const size_t smem = sizeof(int) * ((size_t)p.E * (1 + kGroupThreads / 32) +
                                       (p.path == QMOE_PATH_DECODE ? (size_t)kDtabMax * kDtabInts : 0));
    cudaError_t err = ensure_smem_optin(route_group_small_kernel<4>, 96 * 1024);
    if (err == cudaSuccess) err = ensure_smem_optin(route_group_small_kernel<16>, 96 * 1024);
    if (err != cudaSuccess) return err;
    if (p.E <= 128)
      return launch_pdl(route_group_small_kernel<4>, dim3(1), dim3(kGroupThreads), smem, s, p, xx, lg, ws,
                        x16_mode, (int)want_tiles);
    return launch_pdl(route_group_small_kernel<16>, dim3(1), dim3(kGroupThreads), smem, s, p, xx, lg, ws,
                      x16_mode, (int)want_tiles);
  }
  const int warps = 8;
  int64_t blocks = (p.T + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (p.E <= 128)
    return launch_pdl(route_kernel<4>, dim3((unsigned)blocks), dim3(32 * warps), 0, s, p, xx, lg, ws, x16_mode);
  return launch_pdl(route_kernel<16>, dim3((unsigned)blocks), dim3(32 * warps), 0, s, p, xx, lg, ws, x16_mode);
}

cudaError_t launch_group(const Problem& p, const Workspace& ws, bool want_tiles, cudaStream_t s) {
  if (p.R() <= kPermuteChunk) return cudaSuccess;  // done by route_group_small_kernel
  const unsigned nchunks = (unsigned)ws.nchunks;
  cudaError_t err =
      launch_pdl(group_count_kernel, dim3(nchunks), dim3(kGroupThreads), sizeof(int) * p.E, s, p, ws);
  if (err != cudaSuccess) return err;
  err = launch_pdl(group_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, p, ws, want_tiles ? 1 : 0);
  if (err != cudaSuccess) return err;
  const size_t smem = sizeof(int) * (size_t)p.E * (1 + kGroupThreads / 32);
  return launch_pdl(group_scatter_kernel, dim3(nchunks), dim3(kGroupThreads), smem, s, p, ws);
}

cudaError_t launch_gather(const Problem& p, const Workspace& ws, cudaStream_t s) {
  const int warps = 8;
  int64_t blocks = (p.R() + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(gather_kernel, dim3((unsigned)blocks), dim3(32 * warps), 0, s, p, ws);
}

}  // namespace qmoe
