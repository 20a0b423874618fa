// common.cuh -- device helpers shared by the sm_103a kernels of the MoE layer:
// bf16 unpacking, warp reductions, mbarrier / bulk-copy (TMA) pipeline
// primitives with bounded waits, programmatic dependent launch, and the work
// plan records shared by host and device.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- status codes
// Same values as moe_status_t in include/moe.h.
constexpr int kStatusOk = 0;
constexpr int kStatusDeviceCheck = 5;
constexpr int kStatusTimeout = 6;

// A pipeline wait gives up after kWaitLimitNs of wall time (or kSpinLimit
// polls, whichever comes first), records kStatusTimeout and returns.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kSpinLimit = 1u << 26;
// Each poll may park the thread for up to this long (woken early when the
// phase completes), so waiting warps do not steal issue slots.
constexpr uint32_t kSuspendHintNs = 100000;

// Persistent expert kernels run this many CTAs per SM.
constexpr int kCtasPerSm = 2;

// ---------------------------------------------------------------- plan layout
// One entry per "work expert": every touched routed expert in ascending id,
// then (if present) the shared expert.  Built on the device after align.
struct WorkExpert {
  int32_t expert;      // routed expert id, or -1 for the shared expert
  int32_t n_tok;       // tokens routed to it (T for the shared expert)
  int32_t pos;         // first sorted position of its slots (h row base)
  int32_t unit_gu;     // first gate_up work unit
  int32_t unit_dn;     // first down work unit
  int32_t pad_[3];
};

// The persistent expert kernels run at most this many CTAs.
constexpr int kMaxGrid = 1024;

// Largest top_k the library accepts.
constexpr int kMaxTopK = 16;

struct Plan {
  int32_t n_work;      // number of WorkExpert entries
  int32_t units_gu;    // total gate_up units
  int32_t units_dn;    // total down units
  int32_t num_post_pad;
  int32_t pad_[4];
};

// ---------------------------------------------------------------- bf16 / math
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float sigmoid(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, kStatusOk, code);
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (after recording
// kStatusTimeout) if the phase did not complete within limit_ns of wall time
// or kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0 && global_timer_ns() - t0 > limit_ns) break;
  }
  record_status(status, kStatusTimeout);
  return false;
}

// ---------------------------------------------------------------- bulk copy
// L2 policies: evict-first for data read once (expert weights), evict-last for
// small data many CTAs re-read (activations).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Global -> shared bulk copy (non-tensor TMA).  dst, src 16-byte aligned; bytes
// a multiple of 16.  Completion is signalled on `bar` as transaction bytes.
// Bulk prefetch of [src, src + bytes) into L2 (no completion to wait for);
// src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------ block scan
// Exclusive scan of V ints per thread over the CTA (blockDim a multiple of 32,
// <= 1024).  scratch: >= 32 * V ints.  Every thread gets the totals.
template <int V>
__device__ __forceinline__ void block_scan(const int (&v)[V], int (&ex)[V], int (&tot)[V], int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    inc[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc[i], o);
      if (lane >= o) inc[i] += n;
    }
    if (lane == 31) scratch[i * 32 + warp] = inc[i];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      int s = lane < nw ? scratch[i * 32 + lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += n;
      }
      scratch[i * 32 + lane] = s;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < V; ++i) {
    ex[i] = (warp ? scratch[i * 32 + warp - 1] : 0) + inc[i] - v[i];
    tot[i] = scratch[i * 32 + nw - 1];
  }
  __syncthreads();
}

// ---------------------------------------------------------------- unit split
// Share of a GEMV stage's estimated cost that the CTAs split among themselves
// statically when the stage has a dynamic tail; the units past it go, one at a
// time, to whichever producer asks first (an atomic ticket), so that a CTA
// whose units ran slower than their estimate takes fewer of them.
constexpr float kStaticShare = 0.85f;

// The down stage's CTAs are launched in index order as the gate_up stage's
// CTAs retire, so a later index starts later (by up to the gate_up stage's
// end spread): without a dynamic tail to absorb that, its static share of the
// cost falls linearly across the grid, from (1 + kDownSkew) to (1 - kDownSkew)
// times the average (timed on the decode layers).
constexpr float kDownSkew = 0.15f;

// The cost split of one stage: CTA c starts where the running cost reaches
// G(c / grid) * share * cost, G(x) = (1 + s) x - s x^2 (s = skew; G(x) = x
// without one); with a tail (share < 1) the tail starts at the cost share *
// cost, without one (share 1) the last CTA ends at the last unit.
__host__ __device__ __forceinline__ int split_target(int c, int grid, int cost, bool tail,
                                                   float skew) {
  const int fcost = tail ? (int)(kStaticShare * (float)cost) : cost;
  const float x = (float)c / (float)grid;
  return min(fcost, (int)(((1.0f + skew) * x - skew * x * x) * (float)fcost));
}

// First unit of the work expert whose estimated costs start at c0 (units from
// u0; n tokens in groups of xt, all full but the last; a unit costs base + tw
// x its tokens, base >= 1) at which the running cost reaches `target`.  Units
// are numbered group-major (unit = grp * tiles + tile) or, with tile_major,
// tile-major (unit = tile * groups + grp).
__host__ __device__ __forceinline__ int unit_at_cost(int target, int c0, int u0, int tiles, int n,
                                                     int xt, int base, int tw, bool tile_major) {
  const int groups = (n + xt - 1) / xt;
  const int nt_last = n - (groups - 1) * xt;
  const int full = base + tw * xt;  // cost of a full group's unit
  const int r = target - c0;
  if (tile_major) {
    const int per_tile = (groups - 1) * full + base + tw * nt_last;
    const int t = min(r / per_tile, tiles - 1);
    const int g = min((r - t * per_tile) / full, groups - 1);
    return u0 + t * groups + g;
  }
  const int per_full = tiles * full;
  int g, t;
  if (groups > 1 && r < (groups - 1) * per_full) {
    g = r / per_full;
    t = (r - g * per_full) / full;
  } else {
    g = groups - 1;
    t = min((r - (groups - 1) * per_full) / (base + tw * nt_last), tiles - 1);
  }
  return u0 + g * tiles + t;
}

// Atomic add at GPU scope with acquire-release semantics: the releasing side of
// an arrival counter (stores ordered before it -- by this thread, or by the
// CTA through a preceding barrier -- are published with it) and the acquiring
// side for the last arrival.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ---------------------------------------------------------------- misc
__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace moe
