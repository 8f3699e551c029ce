/*
 * qmoe_oracle.h -- plain CPU oracle of the QMoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product (the CUDA path behind
 * include/qmoe.h) never calls it, and the two share no code.
 *
 * It computes, slowly and in double precision, what the QMoE operator computes
 * (microsoft/onnxruntime "Document and test packed token inputs for MoE and
 * QMoE", #32522; "[CUDA] Add INT4 and INT3 QMoE CPU/GPU offload support",
 * #33575; "[CUDA] Add MoEPacked CPU/GPU hybrid offload ...", #33973):
 *
 *   1. route: per token, the k largest raw router logits (ties to the lower
 *      expert index), weights = softmax over those k logits;
 *   2. group: stable counting sort of the T*k routes by expert;
 *   3. dequantise: w = (code - zero_point) * scale, one scale per block of
 *      `block` weights along K of every weight row;
 *   4. per route: gu = W1_e x_t, h_i = silu(gu_2i) * gu_2i+1, y = W2_e h;
 *   5. combine: out_t = round_once( sum_j w_tj * y_tj ), j ascending, routes
 *      whose weight is exactly 0 skipped.
 *
 * Every sum is taken in double; the only rounding to 16 bits is the final one
 * (round to nearest even, NaN kept NaN).
 */
#ifndef QMOE_ORACLE_H
#define QMOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };

typedef struct {
  int64_t T;       /* packed tokens */
  int32_t H;       /* hidden */
  int32_t inter;   /* I */
  int32_t E;       /* experts */
  int32_t k;       /* top-k */
  int32_t bits;    /* 2, 3 or 4 */
  int32_t block;   /* block size along K */
  int32_t dtype;   /* ORACLE_BF16 / ORACLE_FP16: x, logits, scales, out */
  int32_t full_softmax; /* 0: weights = softmax over the k selected logits (renormalised);
                           1: normalize_routing_weights = 0, each selected expert's
                           probability under the softmax over all E logits */
  int32_t format;  /* ORACLE_INT: integer codes (code - zp) * scale, scales in dtype;
                      ORACLE_MXFP4 / ORACLE_NVFP4: 4-bit E2M1 codes, 8-bit block scales
                      [N][K/block] (E8M0, block 32 / E4M3, block 16), no zero point */
  const float* g1; /* NVFP4: per-expert FP32 global scale of fc1 [E], or NULL (1.0) */
  const float* g2; /* NVFP4: the same for fc2 */
} oracle_problem;

enum { ORACLE_INT = 0, ORACLE_MXFP4 = 1, ORACLE_NVFP4 = 2 };

/* The FP4 expert formats ("NVFP4 block/global scale semantics", "Execution plan
 * to offload export on CPU for a MoE" review; NVFP4 / MXFP4 QMoE weights in
 * "[CUDA] Add INT4 and INT3 QMoE CPU/GPU offload support" #33575), from the
 * published format definitions:
 *   E2M1 element: sign bit 3, exponent bits 2-1 (bias 1), mantissa bit 0; an
 *     exponent field of 0 is subnormal (mantissa * 0.5);
 *   E8M0 scale (MXFP4, one per 32 elements): 2^(b - 127), b = 255 is NaN;
 *   E4M3 scale (NVFP4, one per 16 elements): sign bit 7, exponent bits 6-3
 *     (bias 7), mantissa bits 2-0, subnormal below, the all-ones pattern NaN,
 *     no infinities; NVFP4 weights are also multiplied by an FP32 global scale
 *     (here one per expert and matmul).
 * w = element * block scale (* global scale). */
double oracle_e2m1(unsigned code);
double oracle_e8m0(unsigned bits);
double oracle_e4m3(unsigned bits);

/* Router logits ahead of routing (the router part of the pages' RouterGateUpProj
 * op, "[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload ..." #33731: one GEMM of
 * the packed tokens with the router weight whose output feeds QMoE as raw
 * logits): logits[t][e] = round( sum_h x[t][h] * w_router[e][h] ), the sum in
 * double over h ascending, rounded once to the problem's dtype. x [T][H] and
 * w_router [E][H] in dtype, logits [T][E] in dtype. Returns nonzero for an
 * invalid problem. */
int oracle_router_logits(const oracle_problem* p, const uint16_t* x, const uint16_t* w_router,
                         uint16_t* logits);

/* 16-bit float <-> double. */
double oracle_bits_to_double(uint16_t bits, int dtype);
uint16_t oracle_round_to_bits(double v, int dtype);

/* Unpack n codes (LSB-first packing) into one code per byte. */
void oracle_unpack(const uint8_t* packed, int bits, int64_t n, uint8_t* codes);

/* Dequantise row `row` of a [rows][K] weight matrix (one expert's block). */
void oracle_dequant_row(const uint8_t* q, const uint16_t* scales, const uint8_t* zp,
                        int bits, int block, int dtype, int K, int64_t row, double* out);

/* Routing of every token: topk_idx [T][k], topk_w [T][k] (double). */
int oracle_route(const oracle_problem* p, const uint16_t* logits, int32_t* topk_idx, double* topk_w);

/* Stable grouping of the T*k routes by expert. */
int oracle_permute(const oracle_problem* p, const int32_t* topk_idx, int32_t* expert_offsets,
                   int32_t* sorted_route, int32_t* route_slot);

/* One expert applied to one input row (double in, double out). gu [2I], h [I], y [H]. */
void oracle_expert_ffn(const oracle_problem* p, const uint8_t* fc1_q, const uint16_t* fc1_s,
                       const uint8_t* fc1_zp, const uint8_t* fc2_q, const uint16_t* fc2_s,
                       const uint8_t* fc2_zp, int expert, const double* x_row, double* gu,
                       double* h, double* y);

/* The same with optional biases in the layer's dtype (NULL: none): fc1_b [E][2I]
 * is added to gate/up before SwiGLU, fc2_b [E][H] to the expert output. */
void oracle_expert_ffn_bias(const oracle_problem* p, const uint8_t* fc1_q, const uint16_t* fc1_s,
                            const uint8_t* fc1_zp, const uint16_t* fc1_b, const uint8_t* fc2_q,
                            const uint16_t* fc2_s, const uint8_t* fc2_zp, const uint16_t* fc2_b,
                            int expert, const double* x_row, double* gu, double* h, double* y);

/*
 * The layer forward for the tokens listed in `tokens` (NULL: all T tokens, in
 * order). out_bits [n][H] receives the rounded outputs, out_acc [n][H] (may be
 * NULL) the double sums before rounding. nthreads <= 0 uses every core of the
 * process affinity mask. Returns 0, or -1 on invalid arguments.
 */
int oracle_forward(const oracle_problem* p, const uint16_t* x, const uint16_t* logits,
                   const uint8_t* fc1_q, const uint16_t* fc1_s, const uint8_t* fc1_zp,
                   const uint8_t* fc2_q, const uint16_t* fc2_s, const uint8_t* fc2_zp,
                   const int64_t* tokens, int64_t n_tokens, uint16_t* out_bits, double* out_acc,
                   int nthreads);

/* oracle_forward with optional biases fc1_b [E][2I] and fc2_b [E][H] (NULL: none). */
int oracle_forward_bias(const oracle_problem* p, const uint16_t* x, const uint16_t* logits,
                        const uint8_t* fc1_q, const uint16_t* fc1_s, const uint8_t* fc1_zp,
                        const uint16_t* fc1_b, const uint8_t* fc2_q, const uint16_t* fc2_s,
                        const uint8_t* fc2_zp, const uint16_t* fc2_b, const int64_t* tokens,
                        int64_t n_tokens, uint16_t* out_bits, double* out_acc, int nthreads);

/* Number of cores in the calling process's affinity mask. */
int oracle_num_cores(void);

#ifdef __cplusplus
}
#endif
#endif
