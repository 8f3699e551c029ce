/*
 * qmoe_oracle.c -- plain CPU oracle of the QMoE layer forward (see qmoe_oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product. Written for clarity:
 * every step is a direct loop over the definition, in double precision, with
 * no blocking, fusion or reordering. Built with -ffp-contract=off so that the
 * results are the same on x86-64 and AArch64 hosts.
 *
 * Sources (microsoft/onnxruntime pull requests, as mirrored on the pages):
 *  - packed token-major input [T, H], raw router logits [T, E], output [T, H];
 *    routing is token-local ("Document and test packed token inputs for MoE
 *    and QMoE" #32522, Description);
 *  - QMoE takes raw logits and applies top-k then softmax over the selected
 *    logits, the PhiMoESparseMoeBlock reference (#32522, review comments);
 *  - SwiGLU contract: fc1 has 2*inter rows, gate/up rows interleaved, unsigned
 *    codes with zero-point code 2^(bits-1) (#33575 description; #33624 "INT3
 *    CUDA test fixture update"; Olive/Mobius producer contract in the #33575
 *    static review);
 *  - scales [N, K/block] row-major per weight row (#33624 review thread,
 *    scales_are_block_major=false);
 *  - the combine keeps the partial sum unrounded and rounds to BF16/FP16 once,
 *    NaN stays NaN, zero-weight routes add nothing (#33973 key change 4 and
 *    review fixes);
 *  - optional FC1 / FC2 biases [E, 2I] and [E, H] in the activation dtype, the
 *    FC2 bias indexed by the route's expert and added before the one rounding
 *    (#33575 commit notes: bias validation, "original-expert-indexed FC2 bias
 *    before FP16/BF16 rounding"); normalize_routing_weights = 0 kept covered by
 *    the tests (#32522 review), read as the weights being the selected experts'
 *    probabilities under the softmax over all E logits, not renormalised.
 */
#define _GNU_SOURCE
#include "qmoe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* 16-bit floating-point formats, from the IEEE 754 binary16 and bfloat16     */
/* definitions (sign, biased exponent, fraction).                            */
/* ------------------------------------------------------------------------- */

double oracle_bits_to_double(uint16_t b, int dtype) {
  if (dtype == ORACLE_BF16) {
    /* bfloat16 is the upper half of a binary32 value */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  int sign = b >> 15;
  int e = (b >> 10) & 0x1F;
  int m = b & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* Round a double to the nearest 16-bit value, ties to even, and encode it. */
uint16_t oracle_round_to_bits(double v, int dtype) {
  const int p = dtype == ORACLE_BF16 ? 8 : 11;      /* significand bits */
  const int emin = dtype == ORACLE_BF16 ? -126 : -14; /* smallest normal exponent */
  const int bias = dtype == ORACLE_BF16 ? 127 : 15;
  const int mbits = p - 1;
  const double maxfin = dtype == ORACLE_BF16 ? ldexp(255.0, 120) : 65504.0;
  const uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
  const uint16_t inf = dtype == ORACLE_BF16 ? 0x7F80 : 0x7C00;
  if (isnan(v)) return (uint16_t)(sign | (dtype == ORACLE_BF16 ? 0x7FC0 : 0x7E00));
  double a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | inf);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);
  e -= 1; /* a in [2^e, 2^(e+1)) */
  if (e < emin) e = emin;
  const double quantum = ldexp(1.0, e - mbits);
  const double r = rint(a / quantum) * quantum; /* default rounding mode: nearest, ties to even */
  if (r > maxfin) return (uint16_t)(sign | inf);
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, emin)) { /* subnormal */
    const uint32_t m = (uint32_t)(r / ldexp(1.0, emin - mbits));
    return (uint16_t)(sign | m);
  }
  int e2;
  (void)frexp(r, &e2);
  e2 -= 1;
  const uint32_t m = (uint32_t)(r / ldexp(1.0, e2 - mbits)) - (1u << mbits);
  return (uint16_t)(sign | ((uint32_t)(e2 + bias) << mbits) | m);
}

/* ------------------------------------------------------------------------- */
/* Codes. Packing is least-significant bits first along K: INT4 has code 2c  */
/* in the low nibble of byte c; INT2 has four codes per byte; INT3 packs      */
/* eight codes into each 3-byte little-endian group, code i at bits 3i..3i+2. */
/* ------------------------------------------------------------------------- */

static inline unsigned code_at(const uint8_t* row, int bits, int64_t kk) {
  if (bits == 4) {
    const uint8_t b = row[kk / 2];
    return (kk % 2) ? (b >> 4) : (b & 0xF);
  }
  if (bits == 2) {
    const uint8_t b = row[kk / 4];
    return (b >> (2 * (kk % 4))) & 0x3;
  }
  /* bits == 3 */
  const int64_t g = kk / 8;
  const uint32_t group = (uint32_t)row[3 * g] | ((uint32_t)row[3 * g + 1] << 8) |
                         ((uint32_t)row[3 * g + 2] << 16);
  return (group >> (3 * (kk % 8))) & 0x7;
}

void oracle_unpack(const uint8_t* packed, int bits, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)code_at(packed, bits, i);
}

/* w[row][kk] = (code - zp) * scale[row][kk / block]; zp NULL means 2^(bits-1). */
void oracle_dequant_row(const uint8_t* q, const uint16_t* scales, const uint8_t* zp, int bits,
                        int block, int dtype, int K, int64_t row, double* out) {
  const uint8_t* qrow = q + row * ((int64_t)K * bits / 8);
  const int nblk = K / block;
  for (int kk = 0; kk < K; ++kk) {
    const int b = kk / block;
    const double s = oracle_bits_to_double(scales[row * nblk + b], dtype);
    const double z = zp ? (double)zp[row * nblk + b] : (double)(1 << (bits - 1));
    out[kk] = ((double)code_at(qrow, bits, kk) - z) * s;
  }
}

/* ------------------------------------------------------------------------- */
/* FP4 expert formats (see qmoe_oracle.h).                                   */
/* ------------------------------------------------------------------------- */

double oracle_e2m1(unsigned code) {
  const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

double oracle_e8m0(unsigned bits) {
  bits &= 0xFF;
  return bits == 0xFF ? NAN : ldexp(1.0, (int)bits - 127);
}

double oracle_e4m3(unsigned bits) {
  bits &= 0xFF;
  const int sign = bits >> 7, e = (bits >> 3) & 0xF, m = bits & 7;
  if (e == 0xF && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* One weight row of an expert matrix in the problem's format: integer codes
 * through oracle_dequant_row, FP4 codes times their block scale (and, NVFP4,
 * the expert's global scale g; NULL means 1). */
static void dequant_row_fmt(const oracle_problem* p, const uint8_t* q, const void* scales, const uint8_t* zp,
                            const float* g, int expert, int K, int64_t row, double* out) {
  if (p->format == ORACLE_INT) {
    oracle_dequant_row(q, (const uint16_t*)scales, zp, p->bits, p->block, p->dtype, K, row, out);
    return;
  }
  const uint8_t* qrow = q + row * ((int64_t)K / 2);
  const uint8_t* s8 = (const uint8_t*)scales;
  const int nblk = K / p->block;
  const double gs = (p->format == ORACLE_NVFP4 && g) ? (double)g[expert] : 1.0;
  for (int kk = 0; kk < K; ++kk) {
    const unsigned sb = s8[row * nblk + kk / p->block];
    const double s = p->format == ORACLE_MXFP4 ? oracle_e8m0(sb) : oracle_e4m3(sb);
    out[kk] = oracle_e2m1(code_at(qrow, 4, kk)) * s * gs;
  }
}

/* ------------------------------------------------------------------------- */
/* Routing                                                                   */
/* ------------------------------------------------------------------------- */

/* Is expert a (logit la) ranked ahead of expert b?  Larger logit first, equal
 * logits (+0 == -0) by lower index, NaN after every number. */
static int ranked_ahead(double la, int a, double lb, int b) {
  const int na = isnan(la), nb = isnan(lb);
  if (na || nb) {
    if (na && nb) return a < b;
    return nb;
  }
  if (la != lb) return la > lb;
  return a < b;
}

static void route_token(const oracle_problem* p, const uint16_t* lrow, int32_t* idx, double* w) {
  const int E = p->E, k = p->k;
  char* taken = (char*)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    double bl = 0.0;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      const double l = oracle_bits_to_double(lrow[e], p->dtype);
      if (best < 0 || ranked_ahead(l, e, bl, best)) {
        best = e;
        bl = l;
      }
    }
    taken[best] = 1;
    idx[j] = best;
  }
  free(taken);
  /* softmax over the k selected logits, shifted by the largest one; with
   * full_softmax the denominator runs over all E logits instead */
  const double l0 = oracle_bits_to_double(lrow[idx[0]], p->dtype);
  double denom = 0.0;
  for (int j = 0; j < k; ++j) {
    w[j] = exp(oracle_bits_to_double(lrow[idx[j]], p->dtype) - l0);
    denom += w[j];
  }
  if (p->full_softmax) {
    denom = 0.0;
    for (int e = 0; e < E; ++e) denom += exp(oracle_bits_to_double(lrow[e], p->dtype) - l0);
  }
  for (int j = 0; j < k; ++j) w[j] /= denom;
}

static int valid_problem(const oracle_problem* p) {
  if (!p || p->T < 0 || p->E <= 0 || p->k <= 0 || p->k > p->E || p->H <= 0 || p->inter <= 0) return 0;
  if (p->bits != 2 && p->bits != 3 && p->bits != 4) return 0;
  if (p->block <= 0 || p->H % p->block || p->inter % p->block) return 0;
  if (p->H % 8 || p->inter % 8) return 0;
  if (p->dtype != ORACLE_BF16 && p->dtype != ORACLE_FP16) return 0;
  if (p->full_softmax != 0 && p->full_softmax != 1) return 0;
  if (p->format != ORACLE_INT && p->format != ORACLE_MXFP4 && p->format != ORACLE_NVFP4) return 0;
  if (p->format != ORACLE_INT && p->bits != 4) return 0;
  return 1;
}

int oracle_route(const oracle_problem* p, const uint16_t* logits, int32_t* topk_idx, double* topk_w) {
  if (!valid_problem(p)) return -1;
  for (int64_t t = 0; t < p->T; ++t)
    route_token(p, logits + t * p->E, topk_idx + t * p->k, topk_w + t * p->k);
  return 0;
}

/* Counting sort of route ids r = t*k + j by expert, stable in r. */
int oracle_permute(const oracle_problem* p, const int32_t* topk_idx, int32_t* expert_offsets,
                   int32_t* sorted_route, int32_t* route_slot) {
  if (!valid_problem(p)) return -1;
  const int64_t R = p->T * p->k;
  int64_t* count = (int64_t*)calloc((size_t)p->E + 1, sizeof(int64_t));
  for (int64_t r = 0; r < R; ++r) count[topk_idx[r]]++;
  int64_t run = 0;
  for (int e = 0; e < p->E; ++e) {
    const int64_t c = count[e];
    expert_offsets[e] = (int32_t)run;
    count[e] = run; /* becomes the write cursor */
    run += c;
  }
  expert_offsets[p->E] = (int32_t)run;
  for (int64_t r = 0; r < R; ++r) {
    const int64_t pos = count[topk_idx[r]]++;
    sorted_route[pos] = (int32_t)r;
    if (route_slot) route_slot[r] = (int32_t)pos;
  }
  free(count);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Expert FFN and the layer                                                  */
/* ------------------------------------------------------------------------- */

/* ------------------------------------------------------------------------- */
/* Router logits: a plain dot product per (token, expert), one rounding.      */
/* ------------------------------------------------------------------------- */

int oracle_router_logits(const oracle_problem* p, const uint16_t* x, const uint16_t* w_router,
                         uint16_t* logits) {
  if (!p || p->T < 0 || p->H <= 0 || p->E <= 0 || !x || !w_router || !logits) return 1;
  for (int64_t t = 0; t < p->T; ++t)
    for (int e = 0; e < p->E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < p->H; ++h)
        acc += oracle_bits_to_double(x[t * p->H + h], p->dtype) *
               oracle_bits_to_double(w_router[(int64_t)e * p->H + h], p->dtype);
      logits[t * p->E + e] = oracle_round_to_bits(acc, p->dtype);
    }
  return 0;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

void oracle_expert_ffn(const oracle_problem* p, const uint8_t* fc1_q, const uint16_t* fc1_s,
                       const uint8_t* fc1_zp, const uint8_t* fc2_q, const uint16_t* fc2_s,
                       const uint8_t* fc2_zp, int expert, const double* x_row, double* gu,
                       double* h, double* y) {
  oracle_expert_ffn_bias(p, fc1_q, fc1_s, fc1_zp, NULL, fc2_q, fc2_s, fc2_zp, NULL, expert, x_row, gu,
                         h, y);
}

void oracle_expert_ffn_bias(const oracle_problem* p, const uint8_t* fc1_q, const uint16_t* fc1_s,
                            const uint8_t* fc1_zp, const uint16_t* fc1_b, const uint8_t* fc2_q,
                            const uint16_t* fc2_s, const uint8_t* fc2_zp, const uint16_t* fc2_b,
                            int expert, const double* x_row, double* gu, double* h, double* y) {
  const int H = p->H, I = p->inter;
  const int64_t rows1 = 2 * (int64_t)I, rows2 = H;
  double* wrow = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
  /* fc1: 2I rows of length H; row 2i is gate_i, row 2i+1 is up_i */
  for (int64_t n = 0; n < rows1; ++n) {
    dequant_row_fmt(p, fc1_q, fc1_s, fc1_zp, p->g1, expert, H, (int64_t)expert * rows1 + n, wrow);
    double acc = 0.0;
    for (int kk = 0; kk < H; ++kk) acc += wrow[kk] * x_row[kk];
    if (fc1_b) acc += oracle_bits_to_double(fc1_b[(int64_t)expert * rows1 + n], p->dtype);
    gu[n] = acc;
  }
  for (int i = 0; i < I; ++i) h[i] = silu(gu[2 * i]) * gu[2 * i + 1];
  /* fc2: H rows of length I */
  for (int64_t m = 0; m < rows2; ++m) {
    dequant_row_fmt(p, fc2_q, fc2_s, fc2_zp, p->g2, expert, I, (int64_t)expert * rows2 + m, wrow);
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += wrow[i] * h[i];
    if (fc2_b) acc += oracle_bits_to_double(fc2_b[(int64_t)expert * rows2 + m], p->dtype);
    y[m] = acc;
  }
  free(wrow);
}

typedef struct {
  const oracle_problem* p;
  const uint16_t *x, *logits, *fc1_s, *fc2_s, *fc1_b, *fc2_b;
  const uint8_t *fc1_q, *fc1_zp, *fc2_q, *fc2_zp;
  const int64_t* tokens;
  int64_t n;
  uint16_t* out_bits;
  double* out_acc;
  int64_t next; /* shared work counter */
} fwd_job;

static void forward_token(const fwd_job* J, int64_t slot, double* xr, double* gu, double* h,
                          double* y, double* acc, int32_t* idx, double* w) {
  const oracle_problem* p = J->p;
  const int H = p->H;
  const int64_t t = J->tokens ? J->tokens[slot] : slot;
  route_token(p, J->logits + t * p->E, idx, w);
  for (int kk = 0; kk < H; ++kk) xr[kk] = oracle_bits_to_double(J->x[t * H + kk], p->dtype);
  for (int m = 0; m < H; ++m) acc[m] = 0.0;
  for (int j = 0; j < p->k; ++j) {
    if (w[j] == 0.0) continue; /* a zero-weight route adds nothing */
    oracle_expert_ffn_bias(p, J->fc1_q, J->fc1_s, J->fc1_zp, J->fc1_b, J->fc2_q, J->fc2_s, J->fc2_zp,
                           J->fc2_b, idx[j], xr, gu, h, y);
    for (int m = 0; m < H; ++m) acc[m] += w[j] * y[m];
  }
  for (int m = 0; m < H; ++m) {
    J->out_bits[slot * H + m] = oracle_round_to_bits(acc[m], p->dtype);
    if (J->out_acc) J->out_acc[slot * H + m] = acc[m];
  }
}

static void* forward_worker(void* arg) {
  fwd_job* J = (fwd_job*)arg;
  const oracle_problem* p = J->p;
  const int H = p->H, I = p->inter;
  double* xr = (double*)malloc(sizeof(double) * (size_t)H);
  double* gu = (double*)malloc(sizeof(double) * 2 * (size_t)I);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)p->k);
  double* w = (double*)malloc(sizeof(double) * (size_t)p->k);
  for (;;) {
    const int64_t slot = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (slot >= J->n) break;
    forward_token(J, slot, xr, gu, h, y, acc, idx, w);
  }
  free(xr); free(gu); free(h); free(y); free(acc); free(idx); free(w);
  return NULL;
}

int oracle_num_cores(void) {
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof set, &set) != 0) return 1;
  const int n = CPU_COUNT(&set);
  return n > 0 ? n : 1;
}

int oracle_forward(const oracle_problem* p, const uint16_t* x, const uint16_t* logits,
                   const uint8_t* fc1_q, const uint16_t* fc1_s, const uint8_t* fc1_zp,
                   const uint8_t* fc2_q, const uint16_t* fc2_s, const uint8_t* fc2_zp,
                   const int64_t* tokens, int64_t n_tokens, uint16_t* out_bits, double* out_acc,
                   int nthreads) {
  return oracle_forward_bias(p, x, logits, fc1_q, fc1_s, fc1_zp, NULL, fc2_q, fc2_s, fc2_zp, NULL,
                             tokens, n_tokens, out_bits, out_acc, nthreads);
}

int oracle_forward_bias(const oracle_problem* p, const uint16_t* x, const uint16_t* logits,
                        const uint8_t* fc1_q, const uint16_t* fc1_s, const uint8_t* fc1_zp,
                        const uint16_t* fc1_b, const uint8_t* fc2_q, const uint16_t* fc2_s,
                        const uint8_t* fc2_zp, const uint16_t* fc2_b, const int64_t* tokens,
                        int64_t n_tokens, uint16_t* out_bits, double* out_acc, int nthreads) {
  if (!valid_problem(p) || !out_bits) return -1;
  const int64_t n = tokens ? n_tokens : p->T;
  if (n < 0) return -1;
  if (tokens)
    for (int64_t i = 0; i < n; ++i)
      if (tokens[i] < 0 || tokens[i] >= p->T) return -1;
  if (n == 0) return 0;
  if (!x || !logits || !fc1_q || !fc1_s || !fc2_q || !fc2_s) return -1;
  fwd_job J = {p, x, logits, fc1_s, fc2_s, fc1_b, fc2_b, fc1_q, fc1_zp, fc2_q, fc2_zp, tokens, n,
               out_bits, out_acc, 0};
  int nt = nthreads > 0 ? nthreads : oracle_num_cores();
  if (nt > n) nt = (int)n;
  if (nt <= 1) {
    forward_worker(&J);
    return 0;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  int started = 0;
  for (int i = 0; i < nt; ++i)
    if (pthread_create(&th[i], NULL, forward_worker, &J) == 0) started++;
    else break;
  if (started == 0) forward_worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return 0;
}
