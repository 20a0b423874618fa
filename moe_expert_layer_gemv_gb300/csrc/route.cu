// route.cu -- router GEMV, softmax/top-k/renormalisation, moe_align_block_size
// and the work plan of the grouped expert stages.
//
// Router: logits = x . Wr^T spread over many CTAs (the router fold spread across
// more of the GPU: "veloGB10", Kernel work).  Top-k without a sort: k rounds of
// a warp-wide argmax over the logits held in registers (the sort-free
// verify-path top-k: "Qwen3.8 Flash-Next - GB10 UltraFast", How it works).
// Align: a stable counting sort by expert that keeps arrival order and pads
// every expert to the block size (the moe_align_block_size arrival-order shim:
// same page, What this fork adds), with no atomics, so it is deterministic.
#include <math.h>

#include "launch.h"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;
constexpr int kRouterTokens = 8;  // tokens per router CTA
constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignSmemSlots = 4096;  // routing slots kept in shared memory by align

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  acc = fmaf(bf16lo(a.x), bf16lo(b.x), acc);
  acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
  acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc);
  acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
  acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc);
  acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
  acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc);
  acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
  return acc;
}

// grid = (ceil(E / (8/wpe)), ceil(T / 8)), block = 256.  `wpe` warps share one
// expert row (split along d); each lane holds its CH 16-byte chunks of the row
// in registers, all requested before anything waits; each CTA stages 8 tokens
// of x in shared memory.
template <int CH>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                         float* __restrict__ logits, int T, int d, int E, int wpe) {
  extern __shared__ uint4 xs[];  // [kRouterTokens][d/8]
  __shared__ float red[kRouterWarps][kRouterTokens];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = d >> 3;
  const int t0 = blockIdx.y * kRouterTokens;
  const int nt = min(kRouterTokens, T - t0);
  const int epc = kRouterWarps / wpe;
  const int e = blockIdx.x * epc + warp / wpe;
  const int q = warp % wpe;

  // Router weights are inputs that no kernel of this library writes: request
  // them before waiting on the predecessor.
  const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)min(e, E - 1) * d);
  uint4 w[CH];
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int c = q * 32 + lane + i * wpe * 32;
    w[i] = (e < E && c < nch) ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
  }

  __shared__ __align__(8) uint64_t xbar;
  if (threadIdx.x == 0) {
    mbar_init(&xbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  // The token tile is contiguous: one bulk copy, completion on xbar.
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)nt * d * 2;
    mbar_arrive_expect_tx(&xbar, bytes);
    bulk_g2s(xs, x + (size_t)t0 * d, bytes, &xbar, policy_evict_last());
  }
  const bool ok = mbar_wait(&xbar, 0, nullptr);
  pdl_trigger();
  if (!ok) return;  // unreachable unless the copy never lands; logits are then left unwritten

  float acc[kRouterTokens];
#pragma unroll
  for (int j = 0; j < kRouterTokens; ++j) {
    acc[j] = 0.f;
    if (j < nt) {
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int c = q * 32 + lane + i * wpe * 32;
        if (c < nch) acc[j] = dot8_bf16(w[i], xs[j * nch + c], acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRouterTokens; ++j) acc[j] = warp_sum(acc[j]);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < kRouterTokens; ++j) red[warp][j] = acc[j];
  }
  __syncthreads();
  if (threadIdx.x < epc * kRouterTokens) {
    const int g = threadIdx.x / kRouterTokens, j = threadIdx.x % kRouterTokens;
    const int eo = blockIdx.x * epc + g;
    if (eo < E && j < nt) {
      float s = 0.f;
      for (int p = 0; p < wpe; ++p) s += red[g * wpe + p][j];
      logits[(size_t)(t0 + j) * E + eo] = s;
    }
  }
}

// One warp selects the top-k of one token's E (<= 1024) logits.  Order: larger
// logit first, equal logits -> lower id (softmax is increasing, so this is the
// order of the probabilities).  Weights: exp(l - max) normalised over the
// selected experts (renormalize) or over all E.
template <int NV>
__device__ void warp_topk_nv(const float* __restrict__ L, int E, int k, int renormalize,
                             int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  const int nv = (E + 31) >> 5;
  float v[NV];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    v[i] = -INFINITY;
    const int e = lane + 32 * i;
    if (i < nv && e < E) {
      v[i] = L[e];
      mx = fmaxf(mx, v[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
  if (!renormalize) {
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (i < nv && lane + 32 * i < E) z += expf(v[i] - mx);
    z = warp_sum(z);
  }
  uint32_t taken = 0;
  int my_id = 0;
  float my_e = 0.f, selsum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (i < nv && e < E && !((taken >> i) & 1u) && (bi == 0x7fffffff || v[i] > bv)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    const float ev = expf(bv - mx);
    selsum += ev;
    if (lane == j) {
      my_id = bi;
      my_e = ev;
    }
  }
  out_id = my_id;
  out_w = renormalize ? my_e / selsum : my_e / z;
}

// Dispatch on the number of logits each lane holds (E / 32, rounded up to a
// power of two, E <= 1024).  Lane j < k receives the j-th selected expert and
// its weight.
__device__ void warp_topk(const float* __restrict__ L, int E, int k, int renormalize, int& id,
                          float& wt) {
  const int nv = (E + 31) >> 5;
  if (nv <= 1) warp_topk_nv<1>(L, E, k, renormalize, id, wt);
  else if (nv <= 2) warp_topk_nv<2>(L, E, k, renormalize, id, wt);
  else if (nv <= 4) warp_topk_nv<4>(L, E, k, renormalize, id, wt);
  else if (nv <= 8) warp_topk_nv<8>(L, E, k, renormalize, id, wt);
  else if (nv <= 16) warp_topk_nv<16>(L, E, k, renormalize, id, wt);
  else warp_topk_nv<32>(L, E, k, renormalize, id, wt);
}

// Stores one token's selection (lanes j < k) to its destinations.
__device__ __forceinline__ void store_topk(int k, int id, float wt, int32_t* ids, float* w,
                                           int32_t* ids_copy, float* w_copy, int32_t* ids_smem) {
  const int lane = threadIdx.x & 31;
  if (lane < k) {
    ids[lane] = id;
    w[lane] = wt;
    if (ids_copy) ids_copy[lane] = id;
    if (w_copy) w_copy[lane] = wt;
    if (ids_smem) ids_smem[lane] = id;
  }
}

__global__ void __launch_bounds__(256)
    topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renormalize,
                int32_t* ids, float* w, int32_t* ids_copy, float* w_copy) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  int id;
  float wt;
  warp_topk(logits + (size_t)t * E, E, k, renormalize, id, wt);
  store_topk(k, id, wt, ids + (size_t)t * k, w + (size_t)t * k,
             ids_copy ? ids_copy + (size_t)t * k : nullptr,
             w_copy ? w_copy + (size_t)t * k : nullptr, nullptr);
}

// Exclusive scan of one int per thread over a 1024-thread block.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    scratch[lane] = s;
  }
  __syncthreads();
  const int base = warp ? scratch[warp - 1] : 0;
  *total = scratch[kAlignWarps - 1];
  __syncthreads();
  return base + inc - v;
}

// Estimated cost of a unit with nt tokens, in token-equivalents: a fixed part
// for streaming the unit's weight rows plus one per token of arithmetic.
constexpr int kUnitBaseCost = 4;

// First unit of the CTA whose share of the cost starts at `target`, given
// work expert i's cost prefix `c0`, first unit `u0`, tiles, token count n and
// tokens per group xt (units are numbered group-major).
__device__ int unit_at_cost(int target, int c0, int u0, int tiles, int n, int xt) {
  const int groups = (n + xt - 1) / xt;
  const int nt_last = n - (groups - 1) * xt;
  const int per_full = tiles * (kUnitBaseCost + xt);
  const int r = target - c0;
  int g, t;
  if (groups > 1 && r < (groups - 1) * per_full) {
    g = r / per_full;
    t = (r - g * per_full) / (kUnitBaseCost + xt);
  } else {
    g = groups - 1;
    t = (r - (groups - 1) * per_full) / (kUnitBaseCost + nt_last);
    t = min(t, tiles - 1);
  }
  return u0 + g * tiles + t;
}

// Splits one stage's units over the grid by estimated cost: CTA c gets units
// [cta[c], cta[c+1]) and starts in work expert cta[grid + 1 + c].
__device__ void split_by_cost(int n_work, const int* s_cost, const int* s_unit, const int* s_n,
                              const int* s_tiles, int total_cost, int total_units, int xt,
                              int grid, int32_t* cta) {
  // CTA c's share starts at cost c * total / grid, taken in fp32: monotone in c,
  // and exact enough for balancing (no 64-bit division on the device).
  const float per_cta = (float)total_cost / (float)grid;
  for (int c = threadIdx.x; c <= grid; c += blockDim.x) {
    if (c == grid || n_work == 0) {
      cta[c] = c == grid ? total_units : 0;
      if (c < grid) cta[grid + 1 + c] = 0;
      continue;
    }
    const int target = min(total_cost, (int)((float)c * per_cta));
    int lo = 0, hi = n_work - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_cost[mid] <= target) lo = mid; else hi = mid - 1;
    }
    cta[c] = c == 0 ? 0 : unit_at_cost(target, s_cost[lo], s_unit[lo], s_tiles[lo], s_n[lo], xt);
    cta[grid + 1 + c] = lo;
  }
}

// Work plan: one WorkExpert per touched routed expert (ascending id), then the
// shared expert; gate_up / down work units counted per expert; and each CTA's
// range of units for both expert stages, balanced by estimated cost.  Called by
// all 1024 threads; cnt/off are per-expert counts and padded offsets; tmp holds
// >= 7 * (E + 1) ints of shared memory.
__device__ void build_plan(const int* cnt, const int* off, int E, int T, int num_post_pad,
                           const PlanParams& pp, int* scratch, int* tmp) {
  __syncthreads();
  const int e = threadIdx.x;
  const int c = (e < E) ? cnt[e] : 0;
  const int flag = c > 0;
  const int ggu = (int)ceil_div(c, pp.xt_gu), gdn = (int)ceil_div(c, pp.xt_dn);
  int n_routed, tot_gu, tot_dn, cost_gu, cost_dn;
  const int idx = block_exclusive_scan(flag, scratch, &n_routed);
  const int egu = block_exclusive_scan(flag ? pp.tiles_gu * ggu : 0, scratch, &tot_gu);
  const int edn = block_exclusive_scan(flag ? pp.tiles_dn * gdn : 0, scratch, &tot_dn);
  const int cgu = block_exclusive_scan(
      flag ? pp.tiles_gu * (ggu * kUnitBaseCost + c) : 0, scratch, &cost_gu);
  const int cdn = block_exclusive_scan(
      flag ? pp.tiles_dn * (gdn * kUnitBaseCost + c) : 0, scratch, &cost_dn);
  const int W = E + 1;
  int* s_ugu = tmp;
  int* s_udn = tmp + W;
  int* s_cgu = tmp + 2 * W;
  int* s_cdn = tmp + 3 * W;
  int* s_n = tmp + 4 * W;
  int* s_tgu = tmp + 5 * W;
  int* s_tdn = tmp + 6 * W;
  if (flag) {
    WorkExpert we;
    we.expert = e;
    we.n_tok = c;
    we.pos = off[e];
    we.unit_gu = egu;
    we.unit_dn = edn;
    we.pad_[0] = we.pad_[1] = we.pad_[2] = 0;
    pp.work[idx] = we;
    s_ugu[idx] = egu;
    s_udn[idx] = edn;
    s_cgu[idx] = cgu;
    s_cdn[idx] = cdn;
    s_n[idx] = c;
    s_tgu[idx] = pp.tiles_gu;
    s_tdn[idx] = pp.tiles_dn;
  }
  const bool has_shared = pp.tiles_gu_shared > 0 && T > 0;
  const int n_work = n_routed + (has_shared ? 1 : 0);
  if (has_shared) {
    const int sg = (int)ceil_div(T, pp.xt_gu), sd = (int)ceil_div(T, pp.xt_dn);
    if (threadIdx.x == 0) {
      WorkExpert we;
      we.expert = -1;
      we.n_tok = T;
      we.pos = 0;
      we.unit_gu = tot_gu;
      we.unit_dn = tot_dn;
      we.pad_[0] = we.pad_[1] = we.pad_[2] = 0;
      pp.work[n_routed] = we;
      s_ugu[n_routed] = tot_gu;
      s_udn[n_routed] = tot_dn;
      s_cgu[n_routed] = cost_gu;
      s_cdn[n_routed] = cost_dn;
      s_n[n_routed] = T;
      s_tgu[n_routed] = pp.tiles_gu_shared;
      s_tdn[n_routed] = pp.tiles_dn_shared;
    }
    tot_gu += pp.tiles_gu_shared * sg;
    tot_dn += pp.tiles_dn_shared * sd;
    cost_gu += pp.tiles_gu_shared * (sg * kUnitBaseCost + T);
    cost_dn += pp.tiles_dn_shared * (sd * kUnitBaseCost + T);
  }
  __syncthreads();
  split_by_cost(n_work, s_cgu, s_ugu, s_n, s_tgu, cost_gu, tot_gu, pp.xt_gu, pp.grid,
                pp.cta_gu);
  split_by_cost(n_work, s_cdn, s_udn, s_n, s_tdn, cost_dn, tot_dn, pp.xt_dn, pp.grid,
                pp.cta_dn);
  if (threadIdx.x == 0) {
    Plan p;
    p.n_work = n_work;
    p.units_gu = tot_gu;
    p.units_dn = tot_dn;
    p.num_post_pad = num_post_pad;
    p.pad_[0] = p.pad_[1] = p.pad_[2] = p.pad_[3] = 0;
    *pp.plan = p;
  }
}

// Single CTA of 1024 threads.  Shared memory: hist [32][E] int, cnt [E],
// off [E], scratch [32].
__global__ void __launch_bounds__(kAlignThreads)
    align_kernel(const float* __restrict__ logits, int T, int E, int k, int renormalize,
                 int32_t* ids, float* w, int32_t* ids_copy, float* w_copy, int B,
                 int32_t* __restrict__ sorted_ids, int32_t* __restrict__ block_ids,
                 int32_t* __restrict__ num_post_pad, int32_t* __restrict__ expert_offsets,
                 PlanParams pp, int* status) {
  extern __shared__ int sm[];
  int* hist = sm;                     // [32][E]
  int* cnt = hist + kAlignWarps * E;  // [E]
  int* off = cnt + E;                 // [E]
  int* scratch = off + E;             // [32]
  int* sids = scratch + 32;           // [kAlignSmemSlots] when S fits
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = T * k;
  const bool ids_in_smem = S <= kAlignSmemSlots;

  for (int i = threadIdx.x; i < kAlignWarps * E; i += kAlignThreads) hist[i] = 0;
  pdl_wait();
  pdl_trigger();

  // Optional fused top-k: one warp per token.
  if (logits != nullptr) {
    for (int t = warp; t < T; t += kAlignWarps) {
      int id;
      float wt;
      warp_topk(logits + (size_t)t * E, E, k, renormalize, id, wt);
      store_topk(k, id, wt, ids + (size_t)t * k, w + (size_t)t * k,
                 ids_copy ? ids_copy + (size_t)t * k : nullptr,
                 w_copy ? w_copy + (size_t)t * k : nullptr,
                 ids_in_smem ? sids + (size_t)t * k : nullptr);
    }
  } else if (ids_in_smem) {
    for (int s = threadIdx.x; s < S; s += kAlignThreads) sids[s] = ids[s];
  }
  __syncthreads();
  const int32_t* src = ids_in_smem ? sids : ids;

  // Phase 1: each warp counts the experts of a contiguous chunk of slots.
  const int chunk = (int)ceil_div(S, kAlignWarps);
  const int s_begin = warp * chunk, s_end = min(S, s_begin + chunk);
  for (int base = s_begin; base < s_end; base += 32) {
    const int s = base + lane;
    int e = -1;
    if (s < s_end) {
      e = src[s];
      if (e < 0 || e >= E) {
        record_status(status, kStatusDeviceCheck);
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();

  // Phase 2: per expert, exclusive base of each warp's chunk; totals.
  const int e_me = threadIdx.x;
  int padded = 0;
  if (e_me < E) {
    int run = 0;
    for (int q = 0; q < kAlignWarps; ++q) {
      const int c = hist[q * E + e_me];
      hist[q * E + e_me] = run;
      run += c;
    }
    cnt[e_me] = run;
    padded = (int)round_up(run, B);
  }
  int total;
  const int my_off = block_exclusive_scan(padded, scratch, &total);
  if (e_me < E) {
    off[e_me] = my_off;
    expert_offsets[e_me] = my_off;
    // Pad positions get the sentinel S; every block of the run names e.
    for (int p = my_off + cnt[e_me]; p < my_off + padded; ++p) sorted_ids[p] = S;
    for (int b = my_off / B; b < (my_off + padded) / B; ++b) block_ids[b] = e_me;
  }
  if (threadIdx.x == 0) {
    expert_offsets[E] = total;
    *num_post_pad = total;
  }
  __syncthreads();

  // Phase 3: scatter in arrival order.
  for (int base = s_begin; base < s_end; base += 32) {
    const int s = base + lane;
    int e = -1;
    if (s < s_end) {
      e = src[s];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int rank_base = 0;
    if (e >= 0) rank_base = hist[warp * E + e];
    __syncwarp();
    if (e >= 0) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      sorted_ids[off[e] + rank_base + rank] = s;
      if (lane == __ffs(peers) - 1) hist[warp * E + e] = rank_base + __popc(peers);
    }
    __syncwarp();
  }

  if (pp.work != nullptr) build_plan(cnt, off, E, T, total, pp, scratch, hist);
}

// Plan from an existing align layout: counts recovered from the padded runs
// (a run's trailing entries equal to the sentinel are padding).
__global__ void __launch_bounds__(kAlignThreads)
    plan_kernel(int T, int E, int k, int B, const int32_t* __restrict__ sorted_ids,
                const int32_t* __restrict__ num_post_pad, const int32_t* __restrict__ expert_offsets,
                PlanParams pp, int* status) {
  extern __shared__ int sm[];
  int* cnt = sm;               // [E]
  int* off = cnt + E;          // [E]
  int* scratch = off + E;      // [32]
  int* tmp = scratch + 32;     // [7 * (E + 1)]
  pdl_wait();
  pdl_trigger();
  const int S = T * k;
  const int e = threadIdx.x;
  if (e < E) {
    const int o = expert_offsets[e], o1 = expert_offsets[e + 1];
    const int cap = S + E * (B - 1);
    int c = o1 - o;
    if (o < 0 || c < 0 || c % B != 0 || o1 > cap) {
      record_status(status, kStatusDeviceCheck);
      c = 0;
    }
    int guard = 0;
    while (c > 0 && sorted_ids[o + c - 1] == S && guard++ < B) --c;
    cnt[e] = c;
    off[e] = o;
  }
  __syncthreads();
  build_plan(cnt, off, E, T, *num_post_pad, pp, scratch, tmp);
}

}  // namespace

cudaError_t launch_router_logits(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                                 float* logits, int T, int d, int E, int sms) {
  if (T == 0) return cudaSuccess;
  const int ty = (int)ceil_div(T, kRouterTokens);
  const int nch = d / 8;
  int wpe = 8;
  for (int cand = 1; cand <= 8; cand <<= 1) {
    if (ceil_div(E, kRouterWarps / cand) * ty >= sms) {
      wpe = cand;
      break;
    }
  }
  while (wpe < 8 && ceil_div(nch, wpe * 32) > 8) wpe <<= 1;  // at most 8 chunks per lane
  const int ch = (int)ceil_div(nch, wpe * 32);
  const size_t smem = (size_t)kRouterTokens * d * 2;
  const void* fn = ch <= 1 ? (const void*)router_logits_kernel<1>
                 : ch <= 2 ? (const void*)router_logits_kernel<2>
                 : ch <= 4 ? (const void*)router_logits_kernel<4>
                           : (const void*)router_logits_kernel<8>;
  cudaError_t e = ensure_smem(fn, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(E, kRouterWarps / wpe), (unsigned)ty);
  void* args[] = {&x, &wr, &logits, &T, &d, &E, &wpe};
  return launch_kernel(c, fn, grid, dim3(kRouterWarps * 32), smem, args);
}

cudaError_t launch_topk(const LaunchCfg& c, const float* logits, int T, int E, int k,
                        int renormalize, int32_t* ids, float* w, int32_t* ids_copy,
                        float* w_copy) {
  if (T == 0) return cudaSuccess;
  dim3 grid((unsigned)ceil_div(T, 8));
  void* args[] = {&logits, &T, &E, &k, &renormalize, &ids, &w, &ids_copy, &w_copy};
  return launch_kernel(c, (const void*)topk_kernel, grid, dim3(256), 0, args);
}

cudaError_t launch_align(const LaunchCfg& c, const float* logits, int T, int E, int k,
                         int renormalize, int32_t* ids, float* w, int32_t* ids_copy,
                         float* w_copy, int B, int32_t* sorted_ids, int32_t* block_ids,
                         int32_t* num_post_pad, int32_t* expert_offsets, const PlanParams& pp,
                         int* status) {
  const size_t smem = ((size_t)kAlignWarps * E + 2 * (size_t)E + 32 + kAlignSmemSlots) * sizeof(int);
  cudaError_t e = ensure_smem((const void*)align_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  PlanParams p = pp;
  void* args[] = {&logits, &T, &E, &k, &renormalize, &ids, &w, &ids_copy, &w_copy, &B,
                  &sorted_ids, &block_ids, &num_post_pad, &expert_offsets, &p, &status};
  return launch_kernel(c, (const void*)align_kernel, dim3(1), dim3(kAlignThreads), smem, args);
}

cudaError_t launch_plan(const LaunchCfg& c, int T, int E, int k, int B,
                        const int32_t* sorted_ids, const int32_t* num_post_pad,
                        const int32_t* expert_offsets, const PlanParams& pp, int* status) {
  const size_t smem = (2 * (size_t)E + 32 + 7 * ((size_t)E + 1)) * sizeof(int);
  PlanParams p = pp;
  void* args[] = {&T, &E, &k, &B, &sorted_ids, &num_post_pad, &expert_offsets, &p, &status};
  return launch_kernel(c, (const void*)plan_kernel, dim3(1), dim3(kAlignThreads), smem, args);
}

}  // namespace moe
