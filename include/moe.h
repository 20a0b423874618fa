/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse-MoE expert layer.
 *
 * The layer (one MoE FFN block of a Qwen3.x-style sparse model):
 *   logits[t][e] = x[t] . router_w[e]                          (fp32 accumulate)
 *   p[t]         = softmax_e(logits[t])
 *   ids[t][0..k) = the k largest p, descending, ties -> lower expert id
 *   w[t][j]      = p[t][ids[t][j]] / sum_j' p[t][ids[t][j']]  (renormalised)
 *   h            = silu(W_gate[e] . x[t]) * (W_up[e] . x[t])   (SwiGLU expert)
 *   y[t][j]      = W_down[e] . h
 *   out[t]       = sum_j w[t][j] y[t][j] + sigmoid(x[t] . w_sg) * shared(x[t])
 * Sources: routed experts, top-k and the shared expert -- "veloGB10", The model
 * (512 routed experts, top-10 per token, plus a shared expert) and "How unique
 * is this project? / Kernel work" (router spread across the GPU, grouped MoE
 * expert kernels for decode and prefill that never rebuild full weights, shared
 * expert overlapped with the MoE step, routing folded into neighbouring
 * kernels); the align step with arrival order -- "Qwen3.8 Flash-Next - GB10
 * UltraFast", What this fork adds (moe_align_block_size arrival-order shim);
 * sort-free top-k and W4A16 routed experts -- same page, How it works; int4
 * group size 32 -- same page, Manual.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers to row-major, densely packed
 *     arrays, each 16-byte aligned (checked: MOE_ERR_INVALID_ARG).
 *   - The caller owns every buffer, including the workspace; the library
 *     allocates no device memory.  A workspace is moe_workspace_bytes() bytes,
 *     256-byte aligned, and must be zeroed by moe_workspace_init() once after
 *     allocation.  Calls sharing one workspace must be ordered on one stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous: they enqueue kernels and return; no
 *     call synchronises the host except moe_read_device_status().
 *   - A call may be captured into a CUDA graph (stream capture) once one eager
 *     call with the same dims has run on the device, which sets the kernels'
 *     shared-memory limits; replays then read whatever the captured buffers
 *     hold.
 *   - Every kernel is launched with programmatic dependent launch, the first
 *     of a call included: it may start while the stream's previous kernel
 *     finishes, but it reads no activation, routing or layout input (x, ids,
 *     weights of the combine, align outputs) and writes nothing until that
 *     kernel has completed.  The one exception is router_w: the first kernel
 *     of moe_route / moe_layer_forward requests its router rows before that
 *     wait (every later kernel of a call starts only after the first has
 *     waited).  So the kernel enqueued on the stream just before such a call
 *     must not write router_w; put another kernel, launched without
 *     programmatic dependence, between a router update and the call.
 *     A caller kernel launched programmatically just before a
 *     call must itself wait for its own predecessor (griddepcontrol.wait) if
 *     that predecessor writes this call's inputs.
 *   - Argument errors are detected on the host and returned before anything is
 *     launched.  A failed launch returns MOE_ERR_CUDA.  A kernel that detects a
 *     data-dependent fault (an expert id out of range, a pipeline wait that ran
 *     out of its bound) records a code in the workspace's status word, skips the
 *     bad access and returns; read it with moe_read_device_status().
 *   - bf16 values are IEEE binary32 truncated to their top 16 bits; the output
 *     is rounded to nearest even.
 *   - T == 0: moe_route, moe_expert_forward and moe_layer_forward return MOE_OK
 *     without inspecting any pointer and launch nothing; moe_align_block_size
 *     writes the empty layout (all offsets 0, num_post_pad 0).
 *
 * Limits (MOE_ERR_UNSUPPORTED otherwise): 0 <= T <= 65536, 8 <= d <= 8192 with
 * d % 8 == 0, 1 <= E <= 1024, 1 <= top_k <= min(E, 16), 8 <= I <= 4096 with
 * I % 8 == 0, I_shared == 0 or as I, 1 <= block_size <= 1024.  int4 weights:
 * group_size == 32, d % 256 == 0, I % 256 == 0 (and I_shared % 8 == 0).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad alignment, negative size   */
  MOE_ERR_UNSUPPORTED = 2,  /* dims outside the limits above                */
  MOE_ERR_WORKSPACE = 3,    /* workspace too small or misaligned            */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  MOE_ERR_DEVICE_CHECK = 5, /* a kernel saw an out-of-range routing index   */
  MOE_ERR_TIMEOUT = 6       /* a kernel's bounded pipeline wait ran out     */
} moe_status_t;

typedef enum {
  MOE_WEIGHTS_BF16 = 0,     /* routed experts in bf16                       */
  MOE_WEIGHTS_INT4_G32 = 1  /* symmetric int4, one bf16 scale per 32 values */
} moe_weight_format_t;

/* Bits of moe_dims_t.flags. */
enum {
  /* Batch invariance ("veloGB10", Kernel work: batch-invariant GEMMs, so that a
   * speculative verify pass gives bitwise the result of plain decode steps).
   * Every token's routing (ids, weights) and output row are then bitwise the
   * same whatever the other tokens of the call and whatever T: a token run
   * alone (T = 1) gives the bytes it gets inside any batch.  Without the flag
   * this already holds for T < 256 (the weight-streaming path, whose per-token
   * reduction order is fixed); the flag extends it to every T by keeping
   * prefill-sized calls off the tensor-core GEMMs, which are much faster
   * there but reduce in another order. */
  MOE_FLAG_BATCH_INVARIANT = 1
};

/* Problem dimensions.  T tokens; d model dim; E routed experts; top_k experts
 * per token; I routed-expert intermediate dim; I_shared shared-expert
 * intermediate dim (0 = no shared expert); renormalize (1: weights sum to 1
 * over the selected experts, 0: raw softmax probabilities); block_size = the
 * align block B; weight_format of the ROUTED experts; group_size (int4 only);
 * flags: MOE_FLAG_* bits (0 = none; unknown bits are rejected). */
typedef struct {
  int32_t T, d, E, top_k, I, I_shared;
  int32_t renormalize;
  int32_t block_size;
  int32_t weight_format;
  int32_t group_size;
  int32_t flags;
} moe_dims_t;

/* Routed expert weights (device).
 * BF16:   gate_up bf16 [E][2I][d] (rows [0,I) gate, [I,2I) up);
 *         down bf16 [E][d][I]; both *_scales NULL.
 * INT4_G32: gate_up uint8 [E][2I][d/2], down uint8 [E][d][I/2]: two codes per
 *         byte, even element in the low nibble, stored as code + 8 (0..15);
 *         gate_up_scales bf16 [E][2I][d/32], down_scales bf16 [E][d][I/32].
 *         Element value = (nibble - 8) * scale of its group of 32 along the row
 *         (the reduction dim). */
typedef struct {
  const void* gate_up;
  const void* gate_up_scales;
  const void* down;
  const void* down_scales;
} moe_expert_weights_t;

/* Shared expert (device, bf16): gate_up [2*I_shared][d], down [d][I_shared],
 * gate_w [d] (the sigmoid gate vector w_sg). */
typedef struct {
  const void* gate_up;
  const void* down;
  const void* gate_w;
} moe_shared_weights_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/* Bytes of workspace the calls below need for `dims` (on invalid dims *bytes is
 * 0 and the status says why). */
moe_status_t moe_workspace_bytes(const moe_dims_t* dims, size_t* bytes);

/* Zero a workspace's control words on `stream`: the device status word, the
 * arrival counters of the routing and align kernels (each launch returns its
 * counters to zero) and the work tickets of the two expert GEMV stages (each
 * stage zeroes the other's).  Call once after allocating the workspace, and
 * again if a call left MOE_ERR_TIMEOUT in the status word or failed part-way
 * with MOE_ERR_CUDA (its launches may have stopped short of resetting a
 * counter).  Also disarms moe_workspace_inject_stall. */
moe_status_t moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Byte offsets, from the start of a workspace sized for the same dims, of the
 * routing and aligned layout that moe_layer_forward (and _timed) leave there.
 * Once such a call has completed on its stream, and until the next call that
 * uses the workspace, the regions hold:
 *   topk_ids         int32 [T][top_k]   the call's expert ids
 *   topk_weights     fp32  [T][top_k]   their weights
 *   sorted_ids       int32 [num_post_pad]  moe_align_block_size of those ids
 *   block_expert_ids int32 [num_post_pad / block_size]
 *   num_post_pad     int32 [1]
 *   expert_offsets   int32 [E + 1]
 * with the layout of moe_align_block_size (arrival order, sentinel T*top_k),
 * so a caller can inspect or reuse it (for instance as the layout argument of
 * moe_expert_forward).  Entries past num_post_pad are unspecified.  Host-only:
 * no CUDA call. */
typedef struct {
  size_t topk_ids, topk_weights, sorted_ids, block_expert_ids, num_post_pad, expert_offsets;
} moe_workspace_views_t;
moe_status_t moe_workspace_views(const moe_dims_t* dims, moe_workspace_views_t* views);

/* Test hook for the bounded pipeline waits (the pages' engine fails instead
 * of hanging: "veloGB10", the multi-box section's watchdog).  Arms the
 * workspace so that, in the next layer calls that use it and run the
 * weight-streaming gate_up kernel (every bf16 call below 256 tokens, every
 * int4 call), that kernel's copy-issuing warps issue nothing and its waits give
 * up after about wait_limit_us microseconds (1 ... 1000000) instead of the
 * normal two seconds.  Those calls then record MOE_ERR_TIMEOUT in the status word; their
 * output is unspecified.  No memory is read out of bounds and no kernel faults:
 * the waiting warps simply run out of time.  moe_workspace_init disarms it.
 * Enqueued on `stream` (one 8-byte write into the workspace header). */
moe_status_t moe_workspace_inject_stall(void* workspace, size_t workspace_bytes,
                                        uint32_t wait_limit_us, void* stream);

/* Router GEMV + softmax + top-k + renormalisation ("veloGB10", Kernel work:
 * router spread across the GPU; "Qwen3.8 Flash-Next - GB10 UltraFast", How it
 * works: sort-free top-k).
 *   x bf16 [T][d], router_w bf16 [E][d]
 *   -> topk_ids int32 [T][top_k] (descending probability, ties -> lower id),
 *      topk_weights fp32 [T][top_k].
 * Logits are accumulated in fp32; the softmax uses fp32 expf. */
moe_status_t moe_route(const moe_dims_t* dims, const void* x, const void* router_w,
                       int32_t* topk_ids, float* topk_weights,
                       void* workspace, size_t workspace_bytes, void* stream);

/* moe_align_block_size ("Qwen3.8 Flash-Next - GB10 UltraFast", What this fork
 * adds: the arrival-order shim).  Slots s = t*top_k + j are sorted by expert;
 * within an expert they keep ascending s (arrival order); each expert's run is
 * padded with the sentinel T*top_k to a multiple of block_size.
 *   topk_ids int32 [T*top_k]
 *   -> sorted_ids int32 [T*top_k + E*(block_size-1)] (entries past
 *        num_post_pad are left untouched),
 *      block_expert_ids int32 [(T*top_k + E*(block_size-1)) / block_size + 1]
 *        (expert of each block of block_size sorted positions),
 *      num_post_pad int32 [1] (total padded length),
 *      expert_offsets int32 [E+1] (start of each expert's padded run;
 *        expert_offsets[E] == num_post_pad).
 * Deterministic: no atomics; the same ids give the same bytes. */
moe_status_t moe_align_block_size(const moe_dims_t* dims, const int32_t* topk_ids,
                                  int32_t* sorted_ids, int32_t* block_expert_ids,
                                  int32_t* num_post_pad, int32_t* expert_offsets,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Grouped experts + weighted combine (+ the shared expert when `shared` is not
 * NULL), given the routing and its aligned layout ("veloGB10", Kernel work:
 * grouped MoE expert kernels that never rebuild full weights; shared-expert
 * work overlapped with the MoE step).
 *   x bf16 [T][d]; topk_weights fp32 [T][top_k]; the four align outputs as
 *   produced by moe_align_block_size for the same dims -> out bf16 [T][d].
 * Every slot s < T*top_k must appear exactly once in sorted_ids[0,
 * num_post_pad), inside its expert's run [expert_offsets[e],
 * expert_offsets[e+1]), the run's real slots first and its padding (the
 * sentinel T*top_k) last.  The runs are found from expert_offsets, so
 * block_expert_ids is accepted for the layout's completeness but not read. */
moe_status_t moe_expert_forward(const moe_dims_t* dims, const void* x,
                                const float* topk_weights, const int32_t* sorted_ids,
                                const int32_t* block_expert_ids, const int32_t* num_post_pad,
                                const int32_t* expert_offsets,
                                const moe_expert_weights_t* experts,
                                const moe_shared_weights_t* shared, void* out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer: route, align, experts, combine, shared expert.
 *   x bf16 [T][d], router_w bf16 [E][d] -> out bf16 [T][d].
 *   shared may be NULL (then dims->I_shared must be 0).
 *   topk_ids_out int32 [T][top_k] and topk_weights_out fp32 [T][top_k] are
 *   optional copies of the routing (NULL = not written). */
moe_status_t moe_layer_forward(const moe_dims_t* dims, const void* x, const void* router_w,
                               const moe_expert_weights_t* experts,
                               const moe_shared_weights_t* shared, void* out,
                               int32_t* topk_ids_out, float* topk_weights_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Stage boundaries at which moe_layer_forward_timed records events. */
enum {
  MOE_EV_BEGIN = 0,   /* before the router                            */
  MOE_EV_ROUTED = 1,  /* after router + top-k + align                 */
  MOE_EV_GATE_UP = 2, /* after the gate_up + SwiGLU stage             */
  MOE_EV_DOWN = 3,    /* after the down stage                         */
  MOE_EV_END = 4,     /* after the combine                            */
  MOE_EV_COUNT = 5
};

/* moe_layer_forward, recording events[i] (each a cudaEvent_t passed as void*,
 * created by the caller; a NULL entry is skipped) at the stage boundaries
 * above on `stream`.  The work done is identical to moe_layer_forward. */
moe_status_t moe_layer_forward_timed(const moe_dims_t* dims, const void* x, const void* router_w,
                                     const moe_expert_weights_t* experts,
                                     const moe_shared_weights_t* shared, void* out,
                                     int32_t* topk_ids_out, float* topk_weights_out,
                                     void* workspace, size_t workspace_bytes, void* stream,
                                     void* const* events);

/* Size of the library-owned scratch array used by moe_layer_forward_static. */
#define MOE_STATIC_SCRATCH_BYTES (32u << 20)

/* moe_layer_forward for callers that cannot allocate device memory.  The
 * source pages have no counterpart to this call; it exists for code that may
 * not call cudaMalloc (a caller whose allocator hands out only model tensors, a
 * serving loop that forbids allocation after start-up, a host embedding this
 * library without a caching allocator) and so cannot supply a workspace.
 * Inputs and outputs are still the caller's device buffers, as for
 * moe_layer_forward; the scratch lives in one static device array of
 * MOE_STATIC_SCRATCH_BYTES (32 MiB) inside this library, held by every GPU
 * that loads it until the process exits.  This call allocates nothing.
 *   - Argument errors are returned before anything is enqueued, as for
 *     moe_layer_forward.  Dims whose workspace (moe_workspace_bytes) exceeds
 *     the array are rejected with MOE_ERR_WORKSPACE, also before anything is
 *     enqueued.  Every decode-sized layer of the workloads here fits; a T=4096
 *     prefill layer does not.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     The kept address is not refreshed if the device's primary context is
 *     reset (cudaDeviceReset): do not use this call after such a reset.
 *   - All calls share the one array and each call overwrites it (the status
 *     word is cleared at the start of every call).  Calls that overlap on the
 *     GPU -- on two streams, or from two threads -- race on it and give wrong
 *     results: order them on one stream.
 *   - device_status_out (optional device int32, 4-byte aligned, may be NULL)
 *     receives this call's device status word (MOE_OK or the device-detected
 *     error) at the end of the call, in stream order.
 *   - T == 0 returns MOE_OK at once and, like the other calls, touches
 *     nothing: device_status_out is not written either. */
moe_status_t moe_layer_forward_static(const moe_dims_t* dims, const void* x, const void* router_w,
                                      const moe_expert_weights_t* experts,
                                      const moe_shared_weights_t* shared, void* out,
                                      int32_t* topk_ids_out, float* topk_weights_out,
                                      int32_t* device_status_out, void* stream);

/* Read (and clear) the workspace's device status word.  Synchronises `stream`.
 * *code is MOE_OK or the first device-detected error since the last read. */
moe_status_t moe_read_device_status(void* workspace, int32_t* code, void* stream);

/* Number of this library's kernels enqueued by the calls above since the
 * library was loaded (host-side count; for launch accounting). */
uint64_t moe_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif
