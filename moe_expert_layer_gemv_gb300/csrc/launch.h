// launch.h -- host-side launchers of the MoE layer's kernels (internal to the
// library; the public surface is include/moe.h).  Each launcher enqueues one
// kernel on `stream` and returns the cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "common.cuh"

namespace moe {

// Counts every kernel this library enqueues (moe_kernel_launch_count).
void count_launch();

// Launch attributes: programmatic dependent launch on/off.
struct LaunchCfg {
  cudaStream_t stream;
  bool pdl;  // allow this kernel to start before its predecessor finishes
};

// cudaLaunchKernelExC with the PDL attribute of `c`; counts the launch.
cudaError_t launch_kernel(const LaunchCfg& c, const void* fn, dim3 grid, dim3 block, size_t smem,
                          void** args);

// Sets a kernel's dynamic shared-memory limit once per (device, kernel).
cudaError_t ensure_smem(const void* fn, int bytes);

// Parameters of the work plan built after align (see Plan / WorkExpert).
struct PlanParams {
  WorkExpert* work;      // [E + 1]
  Plan* plan;
  int tiles_gu;          // gate_up tiles per routed expert
  int tiles_dn;          // down tiles per routed expert
  int tiles_gu_shared;   // 0 = no shared expert
  int tiles_dn_shared;
  int xt_gu;             // tokens per gate_up unit
  int xt_dn;             // tokens per down unit
  int base_gu;           // fixed cost of a routed gate_up unit, in tokens of arithmetic
  int base_dn;           // same for down
  int base_gu_s;         // same for the shared expert's (bf16) units
  int base_dn_s;
  int tail_gu, tail_dn;  // 1: the stage ends with a dynamic tail (kStaticShare)
  int tile_major;        // 1: units numbered tile-major (the int4 layers)
  int tok_w;             // cost of a token in a routed unit (0: the tensor-pipe int4
                         // units, whose arithmetic does not grow with their tokens);
                         // a shared-expert unit's tokens cost 1 each
  int tc_nb_gu;          // tensor-core path: N blocks per expert (0 = no tensor-core plan)
  int tc_nb_dn;
  int grid;              // CTAs of the persistent expert kernels (<= kMaxGrid)
  // Per stage: [0, grid] first unit of each CTA (entry grid = total units),
  // then [grid + 1, 2 grid + 1) the work expert each CTA starts in.
  int32_t* cta_gu;
  int32_t* cta_dn;
};

// ------------------------------------------------------------------ routing
// Largest T routed by the single-launch decode path (route_kernel).
constexpr int kFusedRouteMaxT = 128;
// Workspace-header ints used as arrival counters by route_kernel (the status
// word is int 0): [kRouteCounterBase] tiles done, then one per token tile.
constexpr int kRouteCounterBase = 16;
// Workspace-header ints of the GEMV stages' dynamic tails: [kDynCounterBase]
// the gate_up stage's next ticket, [+ 1] the down stage's.  Each stage zeroes
// the other's (zero after moe_workspace_init).
constexpr int kDynCounterBase = 48;
// Workspace-header int counting the finished CTAs of the multi-CTA align.
constexpr int kAlignCounter = 60;
// Workspace-header int holding the stall test hook (moe_workspace_inject_stall):
// 0 = off, else the gate_up stage's wait limit in microseconds, its producers
// issuing nothing.
constexpr int kStallWord = 62;

// *word = value, one thread, in stream order (the stall hook's arming write).
cudaError_t launch_set_word(const LaunchCfg& c, int* word, int value);

// The host-side argument checks of moe_layer_forward other than the workspace:
// dims, pointers, alignment, weights (MOE_OK also for T == 0).
moe_status_t layer_precheck(const moe_dims_t* dims, const void* x, const void* router_w,
                            const moe_expert_weights_t* ex, const moe_shared_weights_t* sh,
                            const void* out, const void* ids_out, const void* w_out);

// logits[t][e] = x[t] . wr[e]; sg[t] = x[t] . w_sg when w_sg (fp32 accumulate).
cudaError_t launch_router_logits(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                                 const uint16_t* w_sg, float* logits, float* sg, int T, int d,
                                 int E, int sms, int* status);

// Whether launch_route_fused handles these dims.
bool fused_route_supported(int T, int E, int k);

// Router + top-k in one launch (decode sizes); with `align`, also the align
// and the workspace plan of the expert stages (by the last token tile).
cudaError_t launch_route_fused(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                               const uint16_t* w_sg, float* logits, float* sg, int T, int d,
                               int E, int k, int renormalize, int32_t* ids, float* w,
                               int32_t* ids_copy, float* w_copy, bool align, int B,
                               int32_t* sorted_ids, int32_t* block_ids, int32_t* num_post_pad,
                               int32_t* expert_offsets, const PlanParams& pp, int* status,
                               int* counters, int sms);

// Per token: softmax over E, top-k (ties -> lower id), (re)normalised weights.
// With w_sg and sg also sg[t] = x[t] . w_sg (fp32, one warp per token).
cudaError_t launch_topk(const LaunchCfg& c, const float* logits, int T, int E, int k,
                        int renormalize, int32_t* ids, float* w, int32_t* ids_copy,
                        float* w_copy, const uint16_t* x, int d, const uint16_t* w_sg, float* sg);

// Single-CTA moe_align_block_size of the given ids, and the work plan when
// pp.work != nullptr.
// S = T * k <= 4096: one CTA.  Larger S: a counting kernel over chunks of
// 1024 slots and a scatter kernel, with chunk_base [E][align_chunks(T, k)] and
// chunk_rank [S] as scratch and *counter (zero between launches) counting the
// counting kernel's finished CTAs.
int align_chunks(int T, int k);
cudaError_t launch_align(const LaunchCfg& c, const int32_t* ids, int T, int E, int k, int B,
                         int32_t* sorted_ids, int32_t* block_ids, int32_t* num_post_pad,
                         int32_t* expert_offsets, const PlanParams& pp, int* status,
                         int32_t* chunk_base, int32_t* chunk_rank, int* counter);

// Work plan from an existing align layout (moe_expert_forward path).
cudaError_t launch_plan(const LaunchCfg& c, int T, int E, int k, int B,
                        const int32_t* sorted_ids, const int32_t* num_post_pad,
                        const int32_t* expert_offsets, const PlanParams& pp, int* status);

// ------------------------------------------------------------------ experts
struct GemvShape {
  int rg;        // gate_up: (gate, up) row pairs per tile  | down: rows per tile (routed)
  int rg_shared; // same for the shared expert
  int xt;        // tokens per unit
  int stage_bytes;
  int n_stages;
  int stage_off; // shared-memory offset of the stage ring
};

// Source of a stage's plan.  ids == nullptr: the plan the align step wrote to
// the workspace (Plan, WorkExpert list, per-CTA unit ranges).  Otherwise
// (decode sizes) every CTA builds the plan in its own shared memory from the
// routing ids; the down stage also writes the aligned layout to the workspace.
struct SmemPlanArgs {
  const int32_t* ids;         // [T*k] routing ids, or nullptr
  int E, B;                   // experts, align block size
  int base, base_s;           // unit cost bases of this stage: routed, shared expert
  int tok_w;                  // cost of a token in a routed unit (shared-expert units: 1)
  int tile_major;             // 1: units numbered tile-major (unit_at_cost)
  int tail;                   // 1: the stage ends with a dynamic tail (kStaticShare)
  int32_t* sorted_ids;        // align outputs to write (down stage), or nullptr
  int32_t* block_ids;
  int32_t* num_post_pad;
  int32_t* expert_offsets;
};

// Persistent shared memory of the shared-memory plan (E experts, S = T*k
// slots), and whether its scratch fits a stage ring of shape g.
int smem_plan_bytes(int E, int S);
bool smem_plan_fits(const GemvShape& g, int E, int T, int k);

struct ExpertArgs {
  int fmt;                  // 0 bf16, 1 int4 (routed experts)
  const void* gate_up;      // routed
  const uint16_t* gate_up_scales;
  const void* down;
  const uint16_t* down_scales;
  const uint16_t* s_gate_up;  // shared (bf16), may be null
  const uint16_t* s_down;
  int T, d, E, k, I, Is;
  int h_rows;               // rows of the h buffer (int4 layers: of each of its two bf16 planes)
};

cudaError_t launch_gate_up(const LaunchCfg& c, const ExpertArgs& a, const GemvShape& g,
                           const uint16_t* x, const int32_t* sorted_ids, const Plan* plan,
                           const WorkExpert* work, const int32_t* cta, const SmemPlanArgs& sp,
                           float* h, float* hs, int* status, int grid, bool tail);

cudaError_t launch_down(const LaunchCfg& c, const ExpertArgs& a, const GemvShape& g,
                        const int32_t* sorted_ids, const Plan* plan, const WorkExpert* work,
                        const int32_t* cta, const SmemPlanArgs& sp, const float* h,
                        const float* hs, float* y, float* ys, int* status, int grid, bool tail);

// out[t] = sum_j w[t][j] y[t*k+j] + sigmoid(sg[t]) ys[t]   (bf16, RNE); sg[t] =
// x[t] . w_sg, read from `sg` when given, else computed here.
cudaError_t launch_combine(const LaunchCfg& c, int T, int d, int k, const float* w,
                           const float* y, const float* ys, const float* sg, const uint16_t* x,
                           const uint16_t* w_sg, uint16_t* out);

// A tiled tensor map of rank 2 or 3: dims and box innermost first, strides in
// bytes of dimensions 1.. (any order: a dimension may step by less than the
// one before it), reads past the end return zeros.
bool encode_map(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                CUtensorMapSwizzle swizzle);

// A 2D tensor map over [rows][cols] elements of `elem_bytes` (row-major),
// box {box_cols, box_rows}, the given swizzle; reads past the end return zeros.
bool encode_map_2d(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* base,
                   uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);

// Tensor-core grouped GEMMs (prefill): whether the dims qualify, and one
// stage's launch (down = false: gate_up + SwiGLU into h; true: down into y/ys).
bool tc_supported(int fmt, int d, int I, int Is, int B);
cudaError_t launch_tc(const LaunchCfg& c, bool down, const ExpertArgs& e, const uint16_t* x,
                      const int32_t* sorted_ids, const Plan* plan, const WorkExpert* work,
                      uint16_t* h, int hs0, int h_rows, float* y, float* ys, int* status,
                      int grid);
// Router logits on the tensor cores: logits[t][e] = x[t] . wr[e] (fp32
// accumulate), for E % 64 == 0, d % 64 == 0, T * d < 2^31.
bool tc_router_supported(int T, int d, int E);
cudaError_t launch_tc_router(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                             float* logits, int T, int d, int E, int* status, int sms);

int tc_tiles_per_mblock_gu(int I);
int tc_tiles_per_mblock_dn(int d);

// Host-side tile/stage choices for the two GEMV stages; `reserve` bytes of
// shared memory before the ring hold the shared-memory plan (0: none).
GemvShape gate_up_shape(int fmt, int d, int I, int Is, int smem_budget, int reserve);
GemvShape down_shape(int fmt, int d, int I, int Is, int smem_budget, int reserve);

}  // namespace moe
