/*
 * moe_oracle.c -- plain fp64 CPU oracle of the sparse-MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h): the reference the CUDA path is
 * checked against, never a product path.  Written for a reader to check by eye:
 * one loop per definition, ascending index order, double everywhere.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double moe_oracle_bf16_to_f64(uint16_t bits) {
  /* bf16 is the top half of an IEEE binary32; widening is exact. */
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

void moe_oracle_decode_bf16(size_t n, const uint16_t* in, double* out) {
  for (size_t i = 0; i < n; ++i) out[i] = moe_oracle_bf16_to_f64(in[i]);
}

/* One int4 element: byte c/2 of the row, low nibble for even c, high for odd;
 * stored offset-binary, so the signed code is u - 8; times the bf16 scale of
 * its group of `group` consecutive elements along the row. */
static double int4_elem(const uint8_t* codes, const uint16_t* scales,
                        size_t row, int32_t cols, int32_t group, int32_t c) {
  uint8_t byte = codes[row * (size_t)(cols / 2) + (size_t)(c / 2)];
  int u = (c & 1) ? (byte >> 4) : (byte & 15);
  double s = moe_oracle_bf16_to_f64(
      scales[row * (size_t)(cols / group) + (size_t)(c / group)]);
  return (double)(u - 8) * s;
}

int moe_oracle_dequant_int4(int32_t rows, int32_t cols, int32_t group,
                            const uint8_t* codes, const uint16_t* scales,
                            double* out) {
  if (rows < 0 || cols <= 0 || cols % 2 || group <= 0 || cols % group) return -1;
  for (int32_t r = 0; r < rows; ++r)
    for (int32_t c = 0; c < cols; ++c)
      out[(size_t)r * cols + c] = int4_elem(codes, scales, (size_t)r, cols, group, c);
  return 0;
}

/* One FP8 E4M3 byte: sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 holds the subnormals m * 2^-9; S.1111.111 is NaN; there is no
 * infinity (the OCP 8-bit floating-point format E4M3). */
double moe_oracle_e4m3_to_f64(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* One FP4 E2M1 code (low 4 bits): sign bit, 2 exponent bits with bias 1, 1
 * mantissa bit; exponent 0 holds the subnormal m * 0.5; no NaN or infinity:
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double moe_oracle_e2m1_to_f64(uint8_t code) {
  const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v;
  if (e == 0)
    v = 0.5 * (double)m;
  else
    v = ldexp(1.0 + (double)m / 2.0, e - 1);
  return sign ? -v : v;
}

/* One FP8 element: byte c of the row (E4M3) times the bf16 scale of its group
 * of `group` consecutive elements along the row. */
static double fp8_elem(const uint8_t* codes, const uint16_t* scales, size_t row, int32_t cols,
                       int32_t group, int32_t c) {
  double s = moe_oracle_bf16_to_f64(scales[row * (size_t)(cols / group) + (size_t)(c / group)]);
  return moe_oracle_e4m3_to_f64(codes[row * (size_t)cols + (size_t)c]) * s;
}

/* One NVFP4 element: E2M1 code in byte c/2 of the row (low nibble for even c,
 * high for odd), times the E4M3 scale of its block of `group` consecutive
 * elements, times the matrix's fp32 scale. */
static double nvfp4_elem(const uint8_t* codes, const uint8_t* scales, double global, size_t row,
                         int32_t cols, int32_t group, int32_t c) {
  uint8_t byte = codes[row * (size_t)(cols / 2) + (size_t)(c / 2)];
  uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
  double s = moe_oracle_e4m3_to_f64(scales[row * (size_t)(cols / group) + (size_t)(c / group)]);
  return moe_oracle_e2m1_to_f64(code) * s * global;
}

int moe_oracle_dequant_fp8(int32_t rows, int32_t cols, int32_t group, const uint8_t* codes,
                           const uint16_t* scales, double* out) {
  if (rows < 0 || cols <= 0 || group <= 0 || cols % group) return -1;
  for (int32_t r = 0; r < rows; ++r)
    for (int32_t c = 0; c < cols; ++c)
      out[(size_t)r * cols + c] = fp8_elem(codes, scales, (size_t)r, cols, group, c);
  return 0;
}

int moe_oracle_dequant_nvfp4(int32_t rows, int32_t cols, int32_t group, const uint8_t* codes,
                             const uint8_t* scales, float global, double* out) {
  if (rows < 0 || cols <= 0 || cols % 2 || group <= 0 || cols % group) return -1;
  for (int32_t r = 0; r < rows; ++r)
    for (int32_t c = 0; c < cols; ++c)
      out[(size_t)r * cols + c] =
          nvfp4_elem(codes, scales, (double)global, (size_t)r, cols, group, c);
  return 0;
}

void moe_oracle_router_logits(int32_t T, int32_t d, int32_t E, const double* x,
                              const double* wr, double* logits) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int32_t i = 0; i < d; ++i) acc += x[(size_t)t * d + i] * wr[(size_t)e * d + i];
      logits[(size_t)t * E + e] = acc;
    }
}

/* Softmax over the E logits of one token: p_e = exp(L_e - max) / sum. */
static void softmax_row(int32_t E, const double* L, double* p) {
  double mx = L[0];
  for (int32_t e = 1; e < E; ++e) if (L[e] > mx) mx = L[e];
  double z = 0.0;
  for (int32_t e = 0; e < E; ++e) { p[e] = exp(L[e] - mx); z += p[e]; }
  for (int32_t e = 0; e < E; ++e) p[e] /= z;
}

typedef struct { double key; int32_t id; } keyed_id;

/* Order: larger key first; equal keys -> lower id first. */
static int cmp_desc_then_id(const void* a, const void* b) {
  const keyed_id* u = (const keyed_id*)a;
  const keyed_id* v = (const keyed_id*)b;
  if (u->key > v->key) return -1;
  if (u->key < v->key) return 1;
  return (u->id > v->id) - (u->id < v->id);
}

/* Full sort of one token's experts by (logit descending, id ascending).  The
 * softmax is strictly increasing in the logit, so this is the same order as by
 * probability, without rounding-made ties. */
static void sort_experts(int32_t E, const double* L, keyed_id* order) {
  for (int32_t e = 0; e < E; ++e) { order[e].key = L[e]; order[e].id = e; }
  qsort(order, (size_t)E, sizeof *order, cmp_desc_then_id);
}

int moe_oracle_topk(int32_t T, int32_t E, int32_t k, int32_t renormalize,
                    const double* logits, int32_t* ids, double* w,
                    double* margin, double* probs) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
  keyed_id* order = (keyed_id*)malloc(sizeof(keyed_id) * (size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  if (!order || !p) { free(order); free(p); return -2; }
  for (int32_t t = 0; t < T; ++t) {
    const double* L = logits + (size_t)t * E;
    softmax_row(E, L, p);
    if (probs) memcpy(probs + (size_t)t * E, p, sizeof(double) * (size_t)E);
    sort_experts(E, L, order);
    double z = 0.0;
    for (int32_t j = 0; j < k; ++j) z += p[order[j].id];
    for (int32_t j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = order[j].id;
      w[(size_t)t * k + j] = renormalize ? p[order[j].id] / z : p[order[j].id];
    }
    if (margin) margin[t] = (k < E) ? order[k - 1].key - order[k].key : INFINITY;
  }
  free(order);
  free(p);
  return 0;
}

int moe_oracle_weights_for_ids(int32_t T, int32_t E, int32_t k,
                               int32_t renormalize, const double* logits,
                               const int32_t* ids, double* w) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  if (!p) return -2;
  for (int32_t t = 0; t < T; ++t) {
    softmax_row(E, logits + (size_t)t * E, p);
    double z = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      int32_t e = ids[(size_t)t * k + j];
      if (e < 0 || e >= E) { free(p); return -1; }
      z += p[e];
    }
    for (int32_t j = 0; j < k; ++j) {
      double pe = p[ids[(size_t)t * k + j]];
      w[(size_t)t * k + j] = renormalize ? pe / z : pe;
    }
  }
  free(p);
  return 0;
}

int moe_oracle_align(int32_t S, int32_t E, int32_t B, const int32_t* ids,
                     int32_t* sorted_ids, int32_t* block_expert_ids,
                     int32_t* num_post_pad, int32_t* expert_offsets,
                     int32_t* counts) {
  if (S < 0 || E <= 0 || B <= 0) return -1;
  /* c_e: how many slots went to expert e. */
  for (int32_t e = 0; e < E; ++e) counts[e] = 0;
  for (int32_t s = 0; s < S; ++s) {
    if (ids[s] < 0 || ids[s] >= E) return -1;
    counts[ids[s]] += 1;
  }
  /* off_e = sum over e' < e of ceil(c_e'/B)*B. */
  int32_t off = 0;
  for (int32_t e = 0; e < E; ++e) {
    expert_offsets[e] = off;
    off += (counts[e] + B - 1) / B * B;
  }
  expert_offsets[E] = off;
  *num_post_pad = off;
  /* Every padded position starts as the sentinel S. */
  for (int32_t i = 0; i < off; ++i) sorted_ids[i] = S;
  /* Arrival order: walk s ascending, append to its expert's segment. */
  for (int32_t e = 0; e < E; ++e) counts[e] = 0;
  for (int32_t s = 0; s < S; ++s) {
    int32_t e = ids[s];
    sorted_ids[expert_offsets[e] + counts[e]] = s;
    counts[e] += 1;
  }
  /* Each block of B positions belongs to the expert whose segment holds it. */
  for (int32_t e = 0; e < E; ++e)
    for (int32_t pos = expert_offsets[e]; pos < expert_offsets[e + 1]; pos += B)
      block_expert_ids[pos / B] = e;
  return 0;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

void moe_oracle_swiglu_expert(int32_t d, int32_t I, const double* x,
                              const double* wgu, const double* wd, double* y) {
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  for (int32_t i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int32_t c = 0; c < d; ++c) g += wgu[(size_t)i * d + c] * x[c];
    for (int32_t c = 0; c < d; ++c) u += wgu[(size_t)(I + i) * d + c] * x[c];
    h[i] = silu(g) * u;
  }
  for (int32_t r = 0; r < d; ++r) {
    double acc = 0.0;
    for (int32_t i = 0; i < I; ++i) acc += wd[(size_t)r * I + i] * h[i];
    y[r] = acc;
  }
  free(h);
}

void moe_oracle_combine(int32_t T, int32_t k, int32_t d, const double* w,
                        const double* y, const double* sg_logit,
                        const double* ys, double* out) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int32_t j = 0; j < k; ++j)
        acc += w[(size_t)t * k + j] * y[((size_t)t * k + j) * d + c];
      if (ys) acc += sigmoid(sg_logit[t]) * ys[(size_t)t * d + c];
      out[(size_t)t * d + c] = acc;
    }
}

/* Row `row` (of expert e) of a routed weight matrix with `cols` columns,
 * decoded to double. */
static void expert_row(const moe_oracle_experts* ex, int which, int32_t e, size_t row,
                       int32_t cols, double* dst) {
  const void* base = which ? ex->down : ex->gate_up;
  const void* sc = which ? ex->down_scales : ex->gate_up_scales;
  if (ex->format == MOE_ORACLE_BF16) {
    moe_oracle_decode_bf16((size_t)cols, (const uint16_t*)base + row * cols, dst);
  } else if (ex->format == MOE_ORACLE_INT4) {
    for (int32_t c = 0; c < cols; ++c)
      dst[c] = int4_elem((const uint8_t*)base, (const uint16_t*)sc, row, cols,
                         ex->group, c);
  } else if (ex->format == MOE_ORACLE_FP8) {
    for (int32_t c = 0; c < cols; ++c)
      dst[c] = fp8_elem((const uint8_t*)base, (const uint16_t*)sc, row, cols, ex->group, c);
  } else if (ex->format == MOE_ORACLE_NVFP4) {
    const double global = (double)(which ? ex->down_global : ex->gate_up_global)[e];
    for (int32_t c = 0; c < cols; ++c)
      dst[c] = nvfp4_elem((const uint8_t*)base, (const uint8_t*)sc, global, row, cols,
                          ex->group, c);
  } else {
    memcpy(dst, (const double*)base + row * cols, sizeof(double) * (size_t)cols);
  }
}

/* Expert e's weights as dense double matrices: wgu [2I][d], wd [d][I]. */
static void expert_dense(const moe_oracle_experts* ex, int32_t e, int32_t d,
                         int32_t I, double* wgu, double* wd) {
  for (int32_t r = 0; r < 2 * I; ++r)
    expert_row(ex, 0, e, (size_t)e * 2 * I + r, d, wgu + (size_t)r * d);
  for (int32_t r = 0; r < d; ++r)
    expert_row(ex, 1, e, (size_t)e * d + r, I, wd + (size_t)r * I);
}

int moe_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int moe_oracle_layer(const moe_oracle_dims* dm, const uint16_t* x,
                     const uint16_t* router_w, const moe_oracle_experts* ex,
                     const moe_oracle_shared* sh, const int32_t* ids_override,
                     const int32_t* token_list, int32_t n,
                     double* out, int32_t* ids_out, double* w_out,
                     double* margin_out, double* sg_out, int32_t nthreads) {
  const int32_t T = dm->T, d = dm->d, E = dm->E, k = dm->k, I = dm->I, Is = dm->Is;
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || I <= 0 || Is < 0) return -1;
  if ((ex->format == MOE_ORACLE_INT4 || ex->format == MOE_ORACLE_NVFP4) &&
      (ex->group <= 0 || d % ex->group || I % ex->group || d % 2 || I % 2)) return -1;
  if (ex->format == MOE_ORACLE_FP8 && (ex->group <= 0 || d % ex->group || I % ex->group))
    return -1;
  if (ex->format == MOE_ORACLE_NVFP4 && (!ex->gate_up_global || !ex->down_global)) return -1;
  if (!token_list) n = T;
  if (n < 0) return -1;
  const int use_shared = (sh != NULL && Is > 0);

  /* Router and shared-gate rows decoded once; experts decoded per use. */
  double* wr = (double*)malloc(sizeof(double) * (size_t)E * d);
  double* wsg = use_shared ? (double*)malloc(sizeof(double) * (size_t)d) : NULL;
  double* sgu = use_shared ? (double*)malloc(sizeof(double) * (size_t)2 * Is * d) : NULL;
  double* sdn = use_shared ? (double*)malloc(sizeof(double) * (size_t)d * Is) : NULL;
  if (!wr || (use_shared && (!wsg || !sgu || !sdn))) {
    free(wr); free(wsg); free(sgu); free(sdn);
    return -2;
  }
  moe_oracle_decode_bf16((size_t)E * d, router_w, wr);
  if (use_shared) {
    moe_oracle_decode_bf16((size_t)d, sh->gate_w, wsg);
    moe_oracle_decode_bf16((size_t)2 * Is * d, sh->gate_up, sgu);
    moe_oracle_decode_bf16((size_t)d * Is, sh->down, sdn);
  }

  int status = 0;
#ifdef _OPENMP
  int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
  {
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    double* L = (double*)malloc(sizeof(double) * (size_t)E);
    double* wgu = (double*)malloc(sizeof(double) * (size_t)2 * I * d);
    double* wd = (double*)malloc(sizeof(double) * (size_t)d * I);
    double* y = (double*)malloc(sizeof(double) * (size_t)(k + 1) * d);
    double* w = (double*)malloc(sizeof(double) * (size_t)k);
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    int ok = xt && L && wgu && wd && y && w && ids;
    if (!ok) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = -2;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int32_t q = 0; q < n; ++q) {
      if (!ok) continue;
      int32_t t = token_list ? token_list[q] : q;
      if (t < 0 || t >= T) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
        status = -1;
        continue;
      }
      moe_oracle_decode_bf16((size_t)d, x + (size_t)t * d, xt);
      /* Router GEMV, softmax, top-k, renormalisation, margin. */
      moe_oracle_router_logits(1, d, E, xt, wr, L);
      double margin;
      if (ids_override) {
        memcpy(ids, ids_override + (size_t)t * k, sizeof(int32_t) * (size_t)k);
        if (moe_oracle_weights_for_ids(1, E, k, dm->renormalize, L, ids, w)) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
          status = -1;
          continue;
        }
        double* scratch_w = (double*)malloc(sizeof(double) * (size_t)k);
        int32_t* scratch_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
        moe_oracle_topk(1, E, k, dm->renormalize, L, scratch_ids, scratch_w, &margin, NULL);
        free(scratch_w);
        free(scratch_ids);
      } else {
        moe_oracle_topk(1, E, k, dm->renormalize, L, ids, w, &margin, NULL);
      }
      /* Routed experts, one SwiGLU FFN per slot. */
      for (int32_t j = 0; j < k; ++j) {
        expert_dense(ex, ids[j], d, I, wgu, wd);
        moe_oracle_swiglu_expert(d, I, xt, wgu, wd, y + (size_t)j * d);
      }
      /* Shared expert and its sigmoid gate. */
      double sg = 0.0;
      if (use_shared) {
        for (int32_t c = 0; c < d; ++c) sg += xt[c] * wsg[c];
        moe_oracle_swiglu_expert(d, Is, xt, sgu, sdn, y + (size_t)k * d);
      }
      moe_oracle_combine(1, k, d, w, y, &sg, use_shared ? y + (size_t)k * d : NULL,
                         out + (size_t)q * d);
      if (ids_out) memcpy(ids_out + (size_t)q * k, ids, sizeof(int32_t) * (size_t)k);
      if (w_out) memcpy(w_out + (size_t)q * k, w, sizeof(double) * (size_t)k);
      if (margin_out) margin_out[q] = margin;
      if (sg_out) sg_out[q] = sg;
    }
    free(xt); free(L); free(wgu); free(wd); free(y); free(w); free(ids);
  }
  free(wr); free(wsg); free(sgu); free(sdn);
  return status;
}
