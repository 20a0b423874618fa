/*
 * moe_oracle.h -- plain fp64 CPU oracle of the sparse-MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the correctness reference that the
 * CUDA path is compared against.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg load it.  It shares no code, header,
 * table or helper with the CUDA library, and it never calls it.
 *
 * What it computes (one MoE FFN layer of a Qwen3.x-style sparse model, as served
 * by the pages "Qwen3.6-35B-A3B on NVIDIA GB10", "Qwen3.6-35B-A3B for NInfer",
 * "Qwen3.8 Flash-Next - GB10 UltraFast" and "veloGB10"):
 *   logits  = x . Wr^T                       (router GEMV; veloGB10, "Kernel work")
 *   p       = softmax over all E experts
 *   ids, w  = top-k of p (ties -> lower id), renormalised to sum to 1
 *             (sort-free top-k on the verify path: Flash-Next, "How it works")
 *   layout  = moe_align_block_size: slots sorted by expert in arrival order,
 *             each expert padded to a block multiple
 *             (arrival-order shim: Flash-Next, "What this fork adds")
 *   h       = silu(Wgate . x) * (Wup . x)     per routed slot (SwiGLU expert)
 *   y       = Wdown . h
 *   out     = sum_j w_j y_j + sigmoid(x . w_sg) * shared_expert(x)
 *             (512 routed experts, top-10, plus a shared expert: veloGB10,
 *              "The model"; shared expert overlapped with the MoE step:
 *              veloGB10, "Kernel work")
 *   int4    = symmetric 4-bit codes, one bf16 scale per group of 32 along the
 *             reduction dim (W4A16 routed experts: Flash-Next, "How it works";
 *             group size 32: Flash-Next, "Manual")
 *   fp8     = E4M3 codes, one bf16 scale per group along the reduction dim
 *   nvfp4   = E2M1 codes, one E4M3 scale per block of 16 along the reduction
 *             dim and one fp32 scale per expert matrix (the "NVFP4/FP8
 *             families" of veloGB10's README; the block layouts are not on the
 *             pages: these are the plainest readings, the int4 grouping for
 *             fp8 and the usual 16-element blocks with an FP8 block scale and a
 *             per-tensor scale for NVFP4)
 *
 * Every floating-point step is done in IEEE double.  bf16, int4, E4M3 and
 * E2M1 inputs are decoded exactly.  There is no blocking, fusion or reordering beyond the plain
 * definition: dot products run in ascending index order.
 *
 * Parity pins (each function is checked against something other than itself by
 * the CPU test tier): brute-force subset search for top-k, closed forms for
 * the softmax/renormalisation special cases, a stable library sort for the
 * align layout, a torch fp64 dense SwiGLU for the expert, a dense-mixture
 * restatement and an identity expert for the combine, an independent numpy
 * dequantisation for int4, torch's float8_e4m3fn on all 256 E4M3 codes, the
 * E2M1 value table, and the layer in each quantised format against the same
 * layer on independently dequantised fp64 weights.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Problem dimensions.  T tokens, model dim d, E routed experts, top-k, expert
 * intermediate I, shared-expert intermediate Is (0 = no shared expert). */
typedef struct {
  int32_t T, d, E, k, I, Is;
  int32_t renormalize; /* 1: w_j = p_j / sum_top p ; 0: w_j = p_j */
} moe_oracle_dims;

/* Routed-expert weight storage formats. */
enum {
  MOE_ORACLE_BF16 = 0,
  MOE_ORACLE_INT4 = 1,
  MOE_ORACLE_F64 = 2,
  MOE_ORACLE_FP8 = 3,
  MOE_ORACLE_NVFP4 = 4
};

/* Routed expert weights.
 *   BF16: gate_up uint16 bf16 bits [E][2I][d], down [E][d][I]; scales NULL.
 *   INT4: gate_up uint8 [E][2I][d/2], down uint8 [E][d][I/2]: two codes per
 *         byte, even element in the low nibble, stored offset-binary u = q+8.
 *         gate_up_scales bf16 [E][2I][d/group], down_scales bf16 [E][d][I/group].
 *         Element value = (u - 8) * scale.
 *   F64 : gate_up double [E][2I][d], down double [E][d][I] (test hook).
 *   FP8 : gate_up uint8 E4M3 [E][2I][d], down uint8 [E][d][I];
 *         gate_up_scales bf16 [E][2I][d/group], down_scales bf16 [E][d][I/group].
 *         Element value = e4m3(code) * scale.
 *   NVFP4: gate_up uint8 [E][2I][d/2], down uint8 [E][d][I/2]: two E2M1 codes
 *         per byte, even element in the low nibble; gate_up_scales uint8 E4M3
 *         [E][2I][d/group], down_scales [E][d][I/group]; gate_up_global,
 *         down_global fp32 [E].  Element value = e2m1(code) * e4m3(scale) *
 *         global[expert]. */
typedef struct {
  int32_t format;
  int32_t group;
  const void* gate_up;
  const void* gate_up_scales;
  const void* down;
  const void* down_scales;
  const float* gate_up_global; /* NVFP4 only, else NULL */
  const float* down_global;
} moe_oracle_experts;

/* Shared expert, bf16 bits: gate_up [2Is][d], down [d][Is], gate_w [d]. */
typedef struct {
  const uint16_t* gate_up;
  const uint16_t* down;
  const uint16_t* gate_w;
} moe_oracle_shared;

/* Exact bf16 -> double. */
double moe_oracle_bf16_to_f64(uint16_t bits);

/* Decode n bf16 values to double. */
void moe_oracle_decode_bf16(size_t n, const uint16_t* in, double* out);

/* Dequantise an int4 matrix [rows][cols] (layout as above) to double. */
int moe_oracle_dequant_int4(int32_t rows, int32_t cols, int32_t group,
                            const uint8_t* codes, const uint16_t* scales,
                            double* out);
/* Exact E4M3 byte -> double (NaN for S.1111.111). */
double moe_oracle_e4m3_to_f64(uint8_t b);
/* Exact E2M1 code (low 4 bits) -> double. */
double moe_oracle_e2m1_to_f64(uint8_t code);
/* Dequantise an FP8 matrix [rows][cols] (layout as above) to double. */
int moe_oracle_dequant_fp8(int32_t rows, int32_t cols, int32_t group, const uint8_t* codes,
                           const uint16_t* scales, double* out);
/* Dequantise an NVFP4 matrix [rows][cols] with matrix scale `global`. */
int moe_oracle_dequant_nvfp4(int32_t rows, int32_t cols, int32_t group, const uint8_t* codes,
                             const uint8_t* scales, float global, double* out);

/* logits[t][e] = sum_i x[t][i] * wr[e][i], ascending i, fp64. */
void moe_oracle_router_logits(int32_t T, int32_t d, int32_t E, const double* x,
                              const double* wr, double* logits);

/* Softmax over E, selection of the k largest (ties -> lower id, output in
 * descending order), renormalisation, and the k-th vs (k+1)-th logit margin
 * (INFINITY when k == E).  probs may be NULL. */
int moe_oracle_topk(int32_t T, int32_t E, int32_t k, int32_t renormalize,
                    const double* logits, int32_t* ids, double* w,
                    double* margin, double* probs);

/* Routing weights for given ids (the override path): w_j from the softmax of
 * that token's logits, renormalised over the given ids when asked. */
int moe_oracle_weights_for_ids(int32_t T, int32_t E, int32_t k,
                               int32_t renormalize, const double* logits,
                               const int32_t* ids, double* w);

/* moe_align_block_size.  S = number of slots (T*k), slot s has expert ids[s].
 *   counts[e]           = #slots routed to e
 *   expert_offsets[e]   = start of e's padded segment, expert_offsets[E] = num_post_pad
 *   sorted_ids[off_e+r] = r-th slot (ascending s) of expert e; pad = S
 *   block_expert_ids[b] = expert owning block b (b < num_post_pad/B)
 * sorted_ids must hold S + E*(B-1) entries, block_expert_ids that / B. */
int moe_oracle_align(int32_t S, int32_t E, int32_t B, const int32_t* ids,
                     int32_t* sorted_ids, int32_t* block_expert_ids,
                     int32_t* num_post_pad, int32_t* expert_offsets,
                     int32_t* counts);

/* One SwiGLU expert on one token: y = Wd . (silu(Wg . x) * (Wu . x)).
 * wgu: [2I][d] rows gate [0,I), up [I,2I); wd: [d][I]; all double. */
void moe_oracle_swiglu_expert(int32_t d, int32_t I, const double* x,
                              const double* wgu, const double* wd, double* y);

/* Combine: out[t] = sum_j w[t][j] * y[t*k+j] + (ys ? sigmoid(sg[t]) * ys[t] : 0).
 * Sum in ascending j, then the shared term. */
void moe_oracle_combine(int32_t T, int32_t k, int32_t d, const double* w,
                        const double* y, const double* sg_logit,
                        const double* ys, double* out);

/* Full layer on a list of tokens (NULL = all T, in order).
 *   x bf16 [T][d], router_w bf16 [E][d]; shared may be NULL.
 *   ids_override [T][k] (may be NULL): route with these ids instead of the
 *     oracle's own selection (weights recomputed from the fp64 softmax).
 *   Outputs are per listed token (n rows): out [n][d]; ids_out [n][k],
 *   w_out [n][k], margin_out [n], sg_out [n] may each be NULL.
 *   nthreads <= 0: OpenMP default. */
int moe_oracle_layer(const moe_oracle_dims* dims, const uint16_t* x,
                     const uint16_t* router_w, const moe_oracle_experts* ex,
                     const moe_oracle_shared* sh, const int32_t* ids_override,
                     const int32_t* token_list, int32_t n,
                     double* out, int32_t* ids_out, double* w_out,
                     double* margin_out, double* sg_out, int32_t nthreads);

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int moe_oracle_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
