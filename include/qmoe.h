/*
 * qmoe.h -- C ABI of the QMoE layer forward on one GB300 (sm_103a).
 *
 * The operator is the quantized Mixture-of-Experts layer of the ONNX Runtime
 * QMoE contrib op as described in the microsoft/onnxruntime pull requests
 * "Document and test packed token inputs for MoE and QMoE" (#32522),
 * "[CUDA] Add INT4 and INT3 QMoE CPU/GPU offload support" (#33575, with the
 * merged texts of #33622, #33629, #33731 and #33624) and "[CUDA] Add MoEPacked
 * CPU/GPU hybrid offload ..." (#33973). For packed token-major input it computes
 *
 *   route   per token t: the top_k largest raw router logits, ties to the lower
 *           expert index, listed by descending logit; weights w[t,j] = softmax
 *           over those top_k logits (#32522: QMoE takes raw logits and applies
 *           top-k then normalisation; reference = softmax over the top-k);
 *   group   the T*top_k routes r = t*top_k + j sorted by expert, stable in r;
 *   fc1     gu = W1_e x_t with W1_e = dequant(fc1_q[e]) of shape [2*inter, hidden],
 *           rows interleaved: row 2i is gate_i, row 2i+1 is up_i (#33575 review:
 *           the producer interleaves gate/up rows and their scales);
 *   swiglu  h_i = silu(gate_i) * up_i, silu(z) = z / (1 + exp(-z))
 *           (activation_type "swiglu", swiglu_fusion = 1; #33624 fixture update);
 *   fc2     y = W2_e h with W2_e = dequant(fc2_q[e]) of shape [hidden, inter];
 *   combine out[t] = round_once( sum_j w[t,j] * y[t*top_k + j] ), j ascending,
 *           FP32 sum, one rounding to the output type, NaN kept NaN, routes with
 *           w == 0 skipped (#33973 key change 4 and review fixes).
 *
 * Dequantisation (#33575 description and #33624 text: unsigned codes, "INT3
 * zero-point code 4", raw layout weights_prepacked = 0, block_size in
 * {32, 64, 128}; #33624 review: scales [N, K/32] row-major):
 *   W[n][kk] = (code[n][kk] - zp[n][kk / block]) * scale[n][kk / block].
 *
 * Layouts (all row-major, all buffers caller-owned device memory):
 *   x            [T][hidden]                        dtype
 *   router_logits[T][num_experts]                   dtype (raw logits)
 *   fc1_q        [E][2*inter][hidden*bits/8]        uint8 packed codes
 *   fc1_scales   [E][2*inter][hidden/block_size]    dtype
 *   fc1_zp       [E][2*inter][hidden/block_size]    uint8, one code per byte, or NULL
 *   fc2_q        [E][hidden][inter*bits/8]          uint8 packed codes
 *   fc2_scales   [E][hidden][inter/block_size]      dtype
 *   fc2_zp       [E][hidden][inter/block_size]      uint8 or NULL
 *   out          [T][hidden]                        dtype
 * Codes are packed least-significant bits first along K as one continuous bit
 * stream: INT4 code 2c is the low nibble of byte c, INT2 has four codes per byte,
 * INT3 eight codes per 3-byte little-endian group (code i at bits 3i..3i+2).
 * A NULL zero-point pointer means the zero point 2^(bits-1) (8, 4 or 2).
 *
 * Precision. Routing compares raw logits exactly; weights use FP32 expf. The
 * expert matmuls run on tensor cores with FP16 operands and FP32 accumulation:
 * dequantised weights (code - zp) * scale are exact in FP16 for BF16 scales in
 * [2^-17, 2^12] (where FP16 scales apply after the MMA, in FP32, any finite
 * scale) and round once for FP16 scales; each token's activations are scaled
 * by a power of two so that their largest magnitude lies in [1, 2) before the
 * FP16 conversion, and the SwiGLU output is stored in FP16 times the square of
 * that power of two and times a power of two set by the expert's first fc1
 * block scale, so that its magnitude does not move with the scale range of the
 * model (parity is tested with BF16 scales from 2^-15 to 2^12, activations with
 * +-1e4 outliers and SwiGLU outputs beyond the FP16 range; an expert whose
 * scales span more than about 2^12 can still leave that range). The combine
 * sums in FP32 and rounds once.
 *
 * Threading and ordering. Every call only enqueues kernels on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and returns; it never
 * synchronises and never copies device to host. The library allocates no
 * memory and keeps no state between calls: all scratch lives in the caller's
 * workspace. Concurrent calls on different streams need distinct workspaces.
 *
 * Errors are returned before any launch, for: null problem or required
 * pointer, T < 0, num_experts <= 0, top_k <= 0, top_k > num_experts, hidden or
 * inter <= 0 (QMOE_ERR_INVALID_ARGUMENT; #33575: validate positive expert and
 * feature dimensions before any arithmetic); bits not in {2,3,4}, block_size
 * not in {32,64,128}, block_size not dividing hidden and inter, hidden or inter
 * not a multiple of 32, num_experts > 512, top_k > 32, unsupported dtype or path
 * (QMOE_ERR_UNSUPPORTED); a pointer that is not 16-byte aligned
 * (QMOE_ERR_MISALIGNED); a workspace smaller than qmoe_workspace_bytes()
 * (QMOE_ERR_WORKSPACE_TOO_SMALL). T == 0 returns QMOE_OK with no launch (#33973:
 * empty input is handled). A failed launch returns QMOE_ERR_CUDA.
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { QMOE_BF16 = 0, QMOE_FP16 = 1 } qmoe_dtype;

typedef enum {
  QMOE_OK = 0,
  QMOE_ERR_INVALID_ARGUMENT = 1,
  QMOE_ERR_UNSUPPORTED = 2,
  QMOE_ERR_MISALIGNED = 3,
  QMOE_ERR_WORKSPACE_TOO_SMALL = 4,
  QMOE_ERR_CUDA = 5
} qmoe_status;

/*
 * Execution path. AUTO takes DECODE for T <= 8 and, up to T = 64 and 512
 * routes (R = T * top_k), while R < 64 or R < 4 * E (the pages switch from their
 * tensor-core GEMV to the grouped GEMM at num_r >= 64 && num_r >= 4 E); GROUPED
 * otherwise.
 * DECODE: weights-stationary dequant-GEMV kernels bound by HBM bandwidth; needs
 * T <= 64, R <= 512 and hidden, inter <= 8192.
 * GROUPED: per-expert dequant-GEMM on tcgen05 tensor cores with TMEM
 * accumulators; needs hidden and inter to be multiples of 64 (bits 2 and 4)
 * or 128 (bits 3). It has two kernels, chosen by the route count: with few
 * routes per expert (R <= 32 * E, and hidden, inter multiples of 256)
 * GROUPED_WS, otherwise GROUPED_ROUTE_TILES.
 * GROUPED_ROUTE_TILES: tiles of 256 sorted routes of one expert on the MMA's M
 * side against 256 (INT3: 128) dequantised weight rows on N.
 * GROUPED_WS (weights-stationary): 128 dequantised weight rows on M against up
 * to 128 routes of one expert on N, in steps of 16; each expert's weights are
 * dequantised once per 128 of its routes, and an expert with a few routes pays
 * for 16-route MMA columns instead of a 128-row route tile. Needs hidden and
 * inter to be multiples of 256 (GROUPED picks route tiles otherwise).
 * The two grouped kernels give results within the same error bound. A path
 * whose condition fails returns QMOE_ERR_UNSUPPORTED.
 */
typedef enum {
  QMOE_PATH_AUTO = 0,
  QMOE_PATH_DECODE = 1,
  QMOE_PATH_GROUPED = 2,
  QMOE_PATH_GROUPED_ROUTE_TILES = 3,
  QMOE_PATH_GROUPED_WS = 4
} qmoe_path;

typedef struct {
  int64_t T;           /* packed tokens (rows of x) */
  int32_t hidden;      /* H */
  int32_t inter;       /* I: SwiGLU width; fc1 has 2*I rows */
  int32_t num_experts; /* E */
  int32_t top_k;       /* k */
  int32_t bits;        /* 2, 3 or 4 */
  int32_t block_size;  /* 32, 64 or 128 weights per scale along K */
  int32_t dtype;       /* qmoe_dtype of x, logits, scales and out */
  int32_t path;        /* qmoe_path */
  int32_t format;      /* qmoe_format of the expert weights (0: integer codes) */
} qmoe_problem;

/*
 * Expert weight formats. QMOE_FORMAT_INT: bits-wide unsigned codes, w = (code -
 * zp) * scale, scales in dtype. The FP4 formats (NVFP4 / MXFP4 QMoE weights,
 * "[CUDA] Add INT4 and INT3 QMoE CPU/GPU offload support" #33575 and the
 * "Execution plan to offload export on CPU for a MoE" review on NVFP4
 * block/global scale semantics) hold 4-bit E2M1 codes (sign bit 3, exponent
 * bits 2-1 with bias 1, mantissa bit 0; values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
 * their negatives), packed like INT4, with one 8-bit block scale per block
 * along K ([E][N][K/block] uint8) and no zero point:
 *   QMOE_FORMAT_MXFP4: block_size 32, E8M0 scales (2^(b - 127); b = 255 is NaN);
 *   QMOE_FORMAT_NVFP4: block_size 16, E4M3 scales (sign, 4 exponent bits with
 *     bias 7, 3 mantissa bits; no infinities, 0x7F / 0xFF NaN), times an FP32
 *     global scale per expert and matmul (qmoe_options.fc1_global_scale /
 *     fc2_global_scale; NULL means 1).
 * w = element * block scale (* global scale). bits must be 4 and the zero-point
 * pointers NULL. The FP4 formats run on both paths. Where hidden and
 * inter are multiples of 256, a call that covers FC1 and FC2 runs them in the
 * decode layer kernel (see qmoe_options.decode_layer_kernel) whatever that
 * option says.
 */
typedef enum { QMOE_FORMAT_INT = 0, QMOE_FORMAT_MXFP4 = 1, QMOE_FORMAT_NVFP4 = 2 } qmoe_format;

/* Bytes of device workspace that qmoe_forward / qmoe_route need for *p
 * (0 if *p is invalid). The same value serves both calls. */
size_t qmoe_workspace_bytes(const qmoe_problem* p);

/*
 * The QMoE layer forward: out = QMoE(x, router_logits, fc1, fc2).
 *
 * Stream order: the call's kernels are launched with programmatic dependent
 * launch, so each may start while the previous kernel on `stream` is still
 * running; every kernel waits for that kernel to complete before it reads
 * anything the previous kernel writes, except that the routing step reads
 * `router_logits` early (the logits are an input the layer never writes). A
 * caller whose own kernel writes `router_logits` directly before this call must
 * therefore not signal early completion to its dependents (a kernel that does not
 * use programmatic launch never does). Results are the same as with plain
 * stream ordering; consecutive calls overlap on the GPU.
 */
qmoe_status qmoe_forward(const qmoe_problem* p, const void* x, const void* router_logits,
                         const uint8_t* fc1_q, const void* fc1_scales, const uint8_t* fc1_zp,
                         const uint8_t* fc2_q, const void* fc2_scales, const uint8_t* fc2_zp,
                         void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Options of qmoe_forward_ex. A zero-filled struct gives qmoe_forward.
 *
 * full_softmax: 0 -- the routing weights are the softmax over the k selected
 *   logits (renormalised over the top-k); 1 -- normalize_routing_weights = 0:
 *   each selected expert's weight is its probability under the softmax over all
 *   E logits of the token, not renormalised ("[CUDA] Document and test packed
 *   token inputs for MoE and QMoE" #32522, review: keep normalize_routing_weights
 *   = 0 covered). A NaN logit anywhere in the row then makes the row's weights NaN.
 * fc1_bias: [E][2*inter] in dtype, row 2j the gate and 2j+1 the up bias of
 *   SwiGLU unit j, added to the fc1 output before SwiGLU; NULL: none.
 * fc2_bias: [E][hidden] in dtype, added to each route's expert output before
 *   the routing weight and the one final rounding; NULL: none ("[CUDA] Add INT4
 *   and INT3 QMoE CPU/GPU offload support" #33575, commit notes: biases
 *   validated as [E, 2*I] and [E, H] in the activation dtype, the FC2 bias
 *   indexed by the route's original expert and applied before the FP16/BF16
 *   rounding).
 * Bias pointers are caller-owned device memory, 16-byte aligned
 * (QMOE_ERR_MISALIGNED otherwise), and only read.
 * decode_layer_kernel: 0 -- one kernel per stage; 1 -- on the decode path
 *   with INT4, block 32, no zero points and hidden, inter multiples of 256,
 *   FC1 and FC2 run as one persistent kernel (the decode layer kernel, whose
 *   warps stream fc1 and fc2 units from one queue); elsewhere the same as 0.
 *   Both give results within the same error bound of the pages' definition;
 *   the layer kernel's result does not depend on the batch a token is packed
 *   into. Other values: QMOE_ERR_INVALID_ARGUMENT.
 * router_weight: [E][hidden] in dtype, caller-owned device memory, 16-byte
 *   aligned, or NULL. When set, the call first computes the router logits from
 *   x (qmoe_router_logits, into the workspace) and routes on them; the
 *   router_logits argument is then not read and may be NULL. The pages run this
 *   GEMM ahead of QMoE as the router part of their RouterGateUpProj op
 *   ("[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload ..." #33731).
 * fc1_global_scale, fc2_global_scale: QMOE_FORMAT_NVFP4 only: FP32 [E] device
 *   arrays (16-byte aligned), the global scale of each expert's fc1 and fc2
 *   weights; NULL means 1. Ignored for the other formats.
 */
typedef struct {
  int32_t full_softmax;
  const void* fc1_bias;
  const void* fc2_bias;
  int32_t decode_layer_kernel;
  const void* router_weight;
  const float* fc1_global_scale;
  const float* fc2_global_scale;
} qmoe_options;

/*
 * qmoe_forward with options (opt may be NULL: the defaults). Extra errors:
 * QMOE_ERR_INVALID_ARGUMENT if opt->full_softmax or opt->decode_layer_kernel
 * is not 0 or 1. The pages
 * define no separate entry point for these options; this one carries them so
 * that qmoe_forward keeps its signature.
 */
qmoe_status qmoe_forward_ex(const qmoe_problem* p, const qmoe_options* opt, const void* x,
                            const void* router_logits, const uint8_t* fc1_q, const void* fc1_scales,
                            const uint8_t* fc1_zp, const uint8_t* fc2_q, const void* fc2_scales,
                            const uint8_t* fc2_zp, void* out, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Stages of qmoe_forward: ROUTE (top-k routing, grouping by expert and the
 * activations' FP16 conversion), FC1 (fc1 dequant-matmul with the SwiGLU
 * epilogue), FC2 (fc2 dequant-matmul, weighted by the routing weight) and
 * COMBINE (sum over each token's routes, rounded once). Each stage runs its
 * own kernels (qmoe_options.decode_layer_kernel = 0).
 */
typedef enum {
  QMOE_STAGE_ROUTE = 0,
  QMOE_STAGE_FC1 = 1,
  QMOE_STAGE_FC2 = 2,
  QMOE_STAGE_COMBINE = 3
} qmoe_stage;

/*
 * Run stages first_stage..last_stage of qmoe_forward (both inclusive). The
 * stages of one forward must be enqueued in order, on one stream, with the same
 * arguments and the same workspace, which carries the intermediate results
 * (routing, grouped activations, SwiGLU output, per-route fc2 output) from one
 * call to the next. qmoe_forward is qmoe_forward_stages(ROUTE, COMBINE). Used
 * to time the stages separately with events between the calls. Returns
 * QMOE_ERR_INVALID_ARGUMENT for a stage range outside ROUTE..COMBINE or with
 * first_stage > last_stage; otherwise the same checks as qmoe_forward.
 */
qmoe_status qmoe_forward_stages(const qmoe_problem* p, int first_stage, int last_stage,
                                const void* x, const void* router_logits, const uint8_t* fc1_q,
                                const void* fc1_scales, const uint8_t* fc1_zp,
                                const uint8_t* fc2_q, const void* fc2_scales,
                                const uint8_t* fc2_zp, void* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Router logits ahead of routing: logits[t][e] = round( sum_h x[t][h] *
 * router_weight[e][h] ), products and sums in FP32 on the tensor cores (BF16 or
 * FP16 operands as given), each logit rounded once to the problem's dtype
 * (nearest even, NaN kept). x [T][hidden], router_weight [E][hidden], logits
 * [T][E], all in dtype, caller-owned device memory, 16-byte aligned. This is
 * the router part of the pages' RouterGateUpProj op, which feeds QMoE its raw
 * logits ("[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload ..." #33731); its
 * gate/up projection belongs to layers outside QMoE and is not computed here.
 * The FP32 sum may differ from an exact one by a unit in the last place of the
 * rounded logit. Uses only the problem's T, hidden, num_experts and dtype (the
 * whole problem is validated as for qmoe_forward). Errors: as qmoe_forward;
 * T == 0 returns QMOE_OK with no launch. Asynchronous on `stream`.
 */
qmoe_status qmoe_router_logits(const qmoe_problem* p, const void* x, const void* router_weight,
                               void* logits, void* stream);

/*
 * Routing and grouping only (the first two steps of qmoe_forward), for
 * inspection and tests: topk_idx int32 [T][k] (descending logit, ties to the
 * lower index), topk_w fp32 [T][k], expert_offsets int32 [E+1] (exclusive
 * prefix of the per-expert route counts), sorted_route int32 [T*k] (route ids
 * t*k+j in expert order, stable in the route id). Any output may be NULL.
 */
qmoe_status qmoe_route(const qmoe_problem* p, const void* router_logits, int32_t* topk_idx,
                       float* topk_w, int32_t* expert_offsets, int32_t* sorted_route,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Static, human-readable name of a status code. */
const char* qmoe_status_string(qmoe_status s);

/*
 * Failure of a kernel after its launch. The pages' own kernels have no such
 * case (they return only argument errors); it exists because every wait inside
 * this library's kernels is bounded in time (about 1 s). A kernel that gives up
 * on a wait writes a nonzero code into an int32 word of the workspace, lets its
 * copies in flight land and returns; the call's last step then writes NaN to
 * every element of `out`, so a failed call never yields plausible numbers.
 * This function returns the byte offset of that word inside a workspace laid
 * out for *p (the same for qmoe_forward, qmoe_forward_ex and the stage calls),
 * or (size_t)-1 when *p is invalid. The word is 0 after a call that completed
 * normally and is reset by the routing step of the next call on the same
 * workspace; read it (for example with cudaMemcpyAsync on the call's stream)
 * after the call and before the next one. Codes: 1 grouped GEMM, 2 decode
 * matmul kernel, 3 decode layer kernel.
 */
size_t qmoe_workspace_error_offset(const qmoe_problem* p);

/*
 * The mixture-of-experts pages have no counterpart of this call: it serves
 * callers that cannot allocate device memory.
 *
 * qmoe_forward on the decode path (T <= 8: path QMOE_PATH_DECODE, or
 * QMOE_PATH_AUTO with T <= 8) with the same arguments, layouts and results,
 * except that the workspace is a fixed device array inside this library of
 * QMOE_STATIC_WORKSPACE_BYTES (8 MiB), which every GPU that loads the library
 * holds until the process exits. The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine); the caller still passes the inputs
 * and `out`. Returns QMOE_ERR_WORKSPACE_TOO_SMALL when qmoe_workspace_bytes(p)
 * exceeds QMOE_STATIC_WORKSPACE_BYTES and QMOE_ERR_UNSUPPORTED when *p resolves
 * to the grouped path; other errors as qmoe_forward. Both checks happen on the
 * host before any CUDA call.
 *
 * The work runs on the calling thread's current device, to which `stream` must
 * belong. The first call with each device and context current looks up the
 * array's device address there (cudaGetSymbolAddress) and caches it for that
 * pair: make that first call before any stream capture on that device, and
 * again after cudaDeviceReset (which creates a new context). All calls on a
 * device share the array, which keeps the previous call's contents; the parts
 * that must start at zero are reset by the call's first kernel. Calls whose
 * GPU work overlaps (different streams or threads without ordering between
 * them) race on the array and give undefined results.
 */
#define QMOE_STATIC_WORKSPACE_BYTES ((size_t)8 << 20)
qmoe_status qmoe_forward_decode_static(const qmoe_problem* p, const void* x,
                                       const void* router_logits, const uint8_t* fc1_q,
                                       const void* fc1_scales, const uint8_t* fc1_zp,
                                       const uint8_t* fc2_q, const void* fc2_scales,
                                       const uint8_t* fc2_zp, void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QMOE_H */
