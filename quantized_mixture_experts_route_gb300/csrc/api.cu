// api.cu -- the C ABI of include/qmoe.h: argument checks, workspace layout and
// the launch sequence of one QMoE layer forward.
//
// Every check happens on the host before any launch (the pages validate
// positive expert and feature dimensions before any arithmetic, "[CUDA] Add
// INT4 and INT3 QMoE CPU/GPU offload support" #33575; empty input is a no-op,
// #33973). The call enqueues work on the caller's stream and returns; it never
// synchronises, allocates or copies device to host.
#include <cstring>

#include "qmoe_internal.cuh"

namespace qmoe {

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

}  // namespace

int resolve_path(const qmoe_problem& p) {
  if (p.path == QMOE_PATH_GROUPED_ROUTE_TILES || p.path == QMOE_PATH_GROUPED_WS) return QMOE_PATH_GROUPED;
  if (p.path != QMOE_PATH_AUTO) return p.path;
  const int64_t R = p.T * (int64_t)p.top_k;
  if (p.T <= 8) return QMOE_PATH_DECODE;
  // mid-size batches: the decode path while the routes are few per expert
  const bool few = R < 64 || R < 4 * (int64_t)p.num_experts;
  return (few && p.T <= kDecodeMaxT && R <= kPermuteChunk) ? QMOE_PATH_DECODE : QMOE_PATH_GROUPED;
}

namespace {

// Shape and attribute checks shared by every entry point.
qmoe_status check_problem(const qmoe_problem* p) {
  if (!p) return QMOE_ERR_INVALID_ARGUMENT;
  if (p->T < 0 || p->num_experts <= 0 || p->top_k <= 0 || p->top_k > p->num_experts ||
      p->hidden <= 0 || p->inter <= 0)
    return QMOE_ERR_INVALID_ARGUMENT;
  if (p->bits != 2 && p->bits != 3 && p->bits != 4) return QMOE_ERR_UNSUPPORTED;
  if (p->format < QMOE_FORMAT_INT || p->format > QMOE_FORMAT_NVFP4) return QMOE_ERR_UNSUPPORTED;
  if (p->format != QMOE_FORMAT_INT) {
    // E2M1 codes with 8-bit block scales: 32 per E8M0 scale, 16 per E4M3 scale
    if (p->bits != 4 || p->block_size != (p->format == QMOE_FORMAT_MXFP4 ? 32 : 16)) return QMOE_ERR_UNSUPPORTED;
  } else if (p->block_size != 32 && p->block_size != 64 && p->block_size != 128) {
    return QMOE_ERR_UNSUPPORTED;
  }
  if (p->hidden % p->block_size || p->inter % p->block_size) return QMOE_ERR_UNSUPPORTED;
  if (p->hidden % 32 || p->inter % 32) return QMOE_ERR_UNSUPPORTED;
  if (p->num_experts > kMaxExperts || p->top_k > kMaxTopK) return QMOE_ERR_UNSUPPORTED;
  if (p->dtype != QMOE_BF16 && p->dtype != QMOE_FP16) return QMOE_ERR_UNSUPPORTED;
  if (p->path < QMOE_PATH_AUTO || p->path > QMOE_PATH_GROUPED_WS) return QMOE_ERR_UNSUPPORTED;
  if ((int64_t)p->T * p->top_k > (int64_t)INT32_MAX / 2) return QMOE_ERR_UNSUPPORTED;
  const int path = resolve_path(*p);
  if (path == QMOE_PATH_DECODE) {
    if (p->T > kDecodeMaxT || p->T * (int64_t)p->top_k > kPermuteChunk) return QMOE_ERR_UNSUPPORTED;
    if (p->hidden > 8192 || p->inter > 8192) return QMOE_ERR_UNSUPPORTED;
  } else {
    const int m = p->bits == 3 ? 128 : 64;
    if (p->hidden % m || p->inter % m) return QMOE_ERR_UNSUPPORTED;
    if (p->path == QMOE_PATH_GROUPED_WS && !grouped_ws_applies(p->hidden, p->inter)) return QMOE_ERR_UNSUPPORTED;
  }
  return QMOE_OK;
}

Problem to_internal(const qmoe_problem& q) {
  Problem p{};
  p.T = q.T;
  p.H = q.hidden;
  p.I = q.inter;
  p.E = q.num_experts;
  p.k = q.top_k;
  p.bits = q.bits;
  p.block = q.block_size;
  p.dtype = q.dtype;
  p.path = resolve_path(q);
  p.format = q.format;
  // the grouped kernel: weights-stationary tiles of kTileWs routes, or route tiles of kTileM
  const int force = q.path == QMOE_PATH_GROUPED_ROUTE_TILES ? 1 : q.path == QMOE_PATH_GROUPED_WS ? 2 : 0;
  p.tile_m = p.path == QMOE_PATH_GROUPED && grouped_ws(p.R(), p.E, p.H, p.I, force) ? kTileWs : kTileM;
  return p;
}

}  // namespace

size_t workspace_layout(const Problem& p, bool grouped, void* base, Workspace* ws) {
  size_t off = 0;
  char* b = static_cast<char*>(base);
  auto take = [&](size_t bytes) -> void* {
    const size_t o = off;
    off += align_up(bytes ? bytes : 1, 256);
    return b ? b + o : nullptr;
  };
  const int64_t R = p.R();
  Workspace w{};
  w.topk_idx = static_cast<int32_t*>(take(sizeof(int32_t) * R));
  w.topk_w = static_cast<float*>(take(sizeof(float) * R));
  w.tok_scale = static_cast<float*>(take(sizeof(float) * p.T));
  w.x16 = static_cast<uint16_t*>(take(sizeof(uint16_t) * p.T * p.H));
  w.offsets = static_cast<int32_t*>(take(sizeof(int32_t) * (p.E + 1)));
  w.sorted_route = static_cast<int32_t*>(take(sizeof(int32_t) * R));
  w.active = static_cast<int32_t*>(take(sizeof(int32_t) * (p.E + kPermuteChunk / kDecodeChunk)));
  w.counters = static_cast<int32_t*>(take(sizeof(int32_t) * 4));
  w.max_tiles = (R + kTileWs - 1) / kTileWs + p.E;   // tiles of either size
  w.tiles = static_cast<int32_t*>(take(sizeof(int32_t) * 2 * w.max_tiles));
  w.nchunks = (R + kPermuteChunk - 1) / kPermuteChunk;
  w.chunk_hist = static_cast<int32_t*>(take(sizeof(int32_t) * w.nchunks * p.E));
  w.dtab = static_cast<int32_t*>(take(sizeof(int32_t) * kDtabInts * kDtabMax));
  const bool dec = p.path == QMOE_PATH_DECODE;
  w.dunits_max = dec ? decode_units_max(p) : 0;
  w.dsplit_items = dec ? decode_split_items_max(p) : 0;
  w.dticket = static_cast<int32_t*>(take(sizeof(int32_t) * w.dunits_max));
  w.dsplit = static_cast<float*>(take(sizeof(float) * 128 * w.dsplit_items));
  w.dsync_ints = dec ? decode_sync_ints(p) : 0;
  w.dsync = static_cast<int32_t*>(take(sizeof(int32_t) * w.dsync_ints));
  w.x16s = grouped ? static_cast<uint16_t*>(take(sizeof(uint16_t) * R * p.H)) : nullptr;
  w.h16 = static_cast<uint16_t*>(take(sizeof(uint16_t) * R * p.I));
  w.y = static_cast<float*>(take(sizeof(float) * R * p.H));
  w.rlogits = static_cast<uint16_t*>(take(sizeof(uint16_t) * p.T * p.E));
  if (ws) *ws = w;
  return off;
}

}  // namespace qmoe

using namespace qmoe;

extern "C" {

size_t qmoe_workspace_bytes(const qmoe_problem* p) {
  if (check_problem(p) != QMOE_OK) return 0;
  const Problem ip = to_internal(*p);
  return workspace_layout(ip, ip.path == QMOE_PATH_GROUPED, nullptr, nullptr);
}

}  // extern "C"

namespace {

qmoe_status forward_impl(const qmoe_problem* p, const qmoe_options* opt, int first_stage, int last_stage,
                         const void* x, const void* router_logits, const uint8_t* fc1_q,
                         const void* fc1_scales, const uint8_t* fc1_zp, const uint8_t* fc2_q,
                         const void* fc2_scales, const uint8_t* fc2_zp, void* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (first_stage < QMOE_STAGE_ROUTE || last_stage > QMOE_STAGE_COMBINE || first_stage > last_stage)
    return QMOE_ERR_INVALID_ARGUMENT;
  const qmoe_status st = check_problem(p);
  if (st != QMOE_OK) return st;
  if (opt && opt->full_softmax != 0 && opt->full_softmax != 1) return QMOE_ERR_INVALID_ARGUMENT;
  if (opt && opt->decode_layer_kernel != 0 && opt->decode_layer_kernel != 1) return QMOE_ERR_INVALID_ARGUMENT;
  if (p->format != QMOE_FORMAT_INT && (fc1_zp || fc2_zp)) return QMOE_ERR_INVALID_ARGUMENT;
  if (p->T == 0) return QMOE_OK;
  // with a router weight the logits are computed from x and the argument is not read
  const void* w_router = opt ? opt->router_weight : nullptr;
  if (w_router) router_logits = w_router;
  if (!x || !router_logits || !fc1_q || !fc1_scales || !fc2_q || !fc2_scales || !out || !workspace)
    return QMOE_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {x, router_logits, fc1_q, fc1_scales, fc2_q, fc2_scales, out, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return QMOE_ERR_MISALIGNED;
  if ((fc1_zp && !aligned16(fc1_zp)) || (fc2_zp && !aligned16(fc2_zp))) return QMOE_ERR_MISALIGNED;
  if (opt && ((opt->fc1_bias && !aligned16(opt->fc1_bias)) || (opt->fc2_bias && !aligned16(opt->fc2_bias))))
    return QMOE_ERR_MISALIGNED;
  if (opt && ((opt->fc1_global_scale && !aligned16(opt->fc1_global_scale)) ||
              (opt->fc2_global_scale && !aligned16(opt->fc2_global_scale))))
    return QMOE_ERR_MISALIGNED;
  Problem ip = to_internal(*p);
  if (opt) {
    ip.full_softmax = opt->full_softmax;
    ip.b1 = static_cast<const uint16_t*>(opt->fc1_bias);
    ip.b2 = static_cast<const uint16_t*>(opt->fc2_bias);
  }
  if (opt && ip.format == QMOE_FORMAT_NVFP4) {
    ip.g1 = opt->fc1_global_scale;
    ip.g2 = opt->fc2_global_scale;
  }
  // the SwiGLU normalisation reads the expert's first fc1 block scale (h_norm)
  ip.s1 = ip.format == QMOE_FORMAT_INT ? static_cast<const uint16_t*>(fc1_scales) : nullptr;
  ip.s1b = ip.format == QMOE_FORMAT_INT ? nullptr : static_cast<const uint8_t*>(fc1_scales);
  const bool grouped = ip.path == QMOE_PATH_GROUPED;
  Workspace ws;
  if (workspace_layout(ip, grouped, workspace, &ws) > workspace_bytes)
    return QMOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto in_range = [&](int stage) { return first_stage <= stage && stage <= last_stage; };
  cudaError_t err = cudaSuccess;
  // FC1 and FC2 of the decode path in one kernel, where it applies: when asked
  // for, and always for the FP4 formats (whose other decode kernel, the generic
  // one, is slower)
  const bool layer_kernel = ((opt && opt->decode_layer_kernel) || ip.format != QMOE_FORMAT_INT) &&
                            in_range(QMOE_STAGE_FC1) && in_range(QMOE_STAGE_FC2) &&
                            decode_layer_applies(ip, fc1_zp || fc2_zp);
  if (in_range(QMOE_STAGE_ROUTE)) {
    if (w_router) {
      err = launch_router_logits(ip, x, w_router, ws.rlogits, s);
      router_logits = ws.rlogits;
      ip.logits_after_wait = 1;
    }
    if (err == cudaSuccess)
      err = launch_route(ip, x, router_logits, ws,
                         decode_int4_blockscaled(ip) ? kX16OddSixteenth
                         : ip.format != QMOE_FORMAT_INT ? kX16Natural : kX16Plain, s);
    if (err == cudaSuccess) err = launch_group(ip, ws, grouped, s);
    if (err == cudaSuccess && grouped) err = launch_gather(ip, ws, s);
  }
  if (err == cudaSuccess && layer_kernel) {
    err = launch_decode_layer(ip, fc1_q, fc1_scales, fc2_q, fc2_scales, ws, s);
    if (err == cudaSuccess && in_range(QMOE_STAGE_COMBINE)) err = launch_combine(ip, ws, out, s);
    if (err == cudaErrorNotSupported) return QMOE_ERR_UNSUPPORTED;
    return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
  }
  if (err == cudaSuccess && in_range(QMOE_STAGE_FC1))
    err = grouped ? launch_grouped(ip, true, fc1_q, fc1_scales, fc1_zp, ws, s)
                  : launch_decode(ip, true, fc1_q, fc1_scales, fc1_zp, ws, s);
  if (err == cudaSuccess && in_range(QMOE_STAGE_FC2))
    err = grouped ? launch_grouped(ip, false, fc2_q, fc2_scales, fc2_zp, ws, s)
                  : launch_decode(ip, false, fc2_q, fc2_scales, fc2_zp, ws, s);
  if (err == cudaSuccess && in_range(QMOE_STAGE_COMBINE)) err = launch_combine(ip, ws, out, s);
  if (err == cudaErrorNotSupported) return QMOE_ERR_UNSUPPORTED;
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

}  // namespace

extern "C" {

qmoe_status qmoe_forward_stages(const qmoe_problem* p, int first_stage, int last_stage,
                                const void* x, const void* router_logits, const uint8_t* fc1_q,
                                const void* fc1_scales, const uint8_t* fc1_zp,
                                const uint8_t* fc2_q, const void* fc2_scales,
                                const uint8_t* fc2_zp, void* out, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return forward_impl(p, nullptr, first_stage, last_stage, x, router_logits, fc1_q, fc1_scales, fc1_zp,
                      fc2_q, fc2_scales, fc2_zp, out, workspace, workspace_bytes, stream);
}

qmoe_status qmoe_forward(const qmoe_problem* p, const void* x, const void* router_logits,
                         const uint8_t* fc1_q, const void* fc1_scales, const uint8_t* fc1_zp,
                         const uint8_t* fc2_q, const void* fc2_scales, const uint8_t* fc2_zp,
                         void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(p, nullptr, QMOE_STAGE_ROUTE, QMOE_STAGE_COMBINE, x, router_logits, fc1_q,
                      fc1_scales, fc1_zp, fc2_q, fc2_scales, fc2_zp, out, workspace, workspace_bytes,
                      stream);
}

qmoe_status qmoe_forward_ex(const qmoe_problem* p, const qmoe_options* opt, const void* x,
                            const void* router_logits, const uint8_t* fc1_q, const void* fc1_scales,
                            const uint8_t* fc1_zp, const uint8_t* fc2_q, const void* fc2_scales,
                            const uint8_t* fc2_zp, void* out, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return forward_impl(p, opt, QMOE_STAGE_ROUTE, QMOE_STAGE_COMBINE, x, router_logits, fc1_q, fc1_scales,
                      fc1_zp, fc2_q, fc2_scales, fc2_zp, out, workspace, workspace_bytes, stream);
}

qmoe_status qmoe_router_logits(const qmoe_problem* p, const void* x, const void* router_weight, void* logits,
                               void* stream) {
  const qmoe_status st = check_problem(p);
  if (st != QMOE_OK) return st;
  if (p->T == 0) return QMOE_OK;
  if (!x || !router_weight || !logits) return QMOE_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(router_weight) || !aligned16(logits)) return QMOE_ERR_MISALIGNED;
  const Problem ip = to_internal(*p);
  const cudaError_t err = launch_router_logits(ip, x, router_weight, logits, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

qmoe_status qmoe_route(const qmoe_problem* p, const void* router_logits, int32_t* topk_idx,
                       float* topk_w, int32_t* expert_offsets, int32_t* sorted_route,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const qmoe_status st = check_problem(p);
  if (st != QMOE_OK) return st;
  if (p->T == 0) return QMOE_OK;
  if (!router_logits || !workspace) return QMOE_ERR_INVALID_ARGUMENT;
  if (!aligned16(router_logits) || !aligned16(workspace)) return QMOE_ERR_MISALIGNED;
  const Problem ip = to_internal(*p);
  const bool grouped = ip.path == QMOE_PATH_GROUPED;
  Workspace ws;
  if (workspace_layout(ip, grouped, workspace, &ws) > workspace_bytes)
    return QMOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = launch_route(ip, nullptr, router_logits, ws, kX16None, s);
  if (err == cudaSuccess) err = launch_group(ip, ws, grouped, s);
  const int64_t R = ip.R();
  if (err == cudaSuccess && topk_idx)
    err = cudaMemcpyAsync(topk_idx, ws.topk_idx, sizeof(int32_t) * R, cudaMemcpyDeviceToDevice, s);
  if (err == cudaSuccess && topk_w)
    err = cudaMemcpyAsync(topk_w, ws.topk_w, sizeof(float) * R, cudaMemcpyDeviceToDevice, s);
  if (err == cudaSuccess && expert_offsets)
    err = cudaMemcpyAsync(expert_offsets, ws.offsets, sizeof(int32_t) * (ip.E + 1),
                          cudaMemcpyDeviceToDevice, s);
  if (err == cudaSuccess && sorted_route)
    err = cudaMemcpyAsync(sorted_route, ws.sorted_route, sizeof(int32_t) * R,
                          cudaMemcpyDeviceToDevice, s);
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

size_t qmoe_workspace_error_offset(const qmoe_problem* p) {
  if (check_problem(p) != QMOE_OK) return (size_t)-1;
  const Problem ip = to_internal(*p);
  Workspace ws;
  // laid out from a nominal base address; nothing is dereferenced
  constexpr uintptr_t kBase = 4096;
  workspace_layout(ip, ip.path == QMOE_PATH_GROUPED, reinterpret_cast<void*>(kBase), &ws);
  return (size_t)(reinterpret_cast<uintptr_t>(ws.counters + 2) - kBase);
}

const char* qmoe_status_string(qmoe_status s) {
  switch (s) {
    case QMOE_OK: return "ok";
    case QMOE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QMOE_ERR_UNSUPPORTED: return "unsupported problem";
    case QMOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case QMOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QMOE_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

}  // extern "C"
