// route.cu -- router GEMV, softmax/top-k/renormalisation, moe_align_block_size
// and the work plan of the grouped expert stages.
//
// Router: logits = x . Wr^T spread over many CTAs (the router fold spread across
// more of the GPU: "veloGB10", Kernel work); the shared expert's gate x . w_sg
// rides along as one more row.  Top-k without a sort: k rounds of a warp-wide
// argmax over the logits held in registers (the sort-free verify-path top-k:
// "Qwen3.8 Flash-Next - GB10 UltraFast", How it works).  Align: a stable
// counting sort by expert that keeps arrival order and pads every expert to the
// block size (the moe_align_block_size arrival-order shim: same page, What this
// fork adds), with no atomics on the data, so it is deterministic.
//
// At decode sizes the whole routing step is one launch (route_kernel): router
// CTAs write logits; the last CTA of each token tile to finish (an integer
// arrival counter) selects that tile's top-k; the last tile to finish runs the
// align and builds the work plan ("veloGB10", Kernel work: the expert routing
// folded into its neighbours).
#include <math.h>

#include "launch.h"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;
constexpr int kRouterThreads = kRouterWarps * 32;
constexpr int kRouterTokens = 8;  // tokens per router CTA (one token tile)
constexpr int kAlignThreads = 1024;
constexpr int kAlignSmemSlots = 4096;  // routing slots the align step keeps in shared memory
constexpr int kScanScratch = 32 * 8;   // ints of scratch for block_scan<V <= 8>

// ------------------------------------------------------------------ router
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

struct RouterArgs {
  const uint16_t* x;       // [T][d]
  const uint16_t* wr;      // [E][d]
  const uint16_t* w_sg;    // [d] shared-expert gate row, or null
  float* logits;           // [T][E]
  float* sg;               // [T] x . w_sg (when w_sg)
  int T, d, E, wpe;
};

// One router CTA: rows [blockIdx.x * epc, +epc) of the E routed rows plus the
// gate row (index E), `wpe` warps per row split along d, one token tile of 8
// tokens staged in shared memory (xs, >= 8 * d bf16) by one bulk copy.  Each
// lane holds its CH 16-byte chunks of its row, requested before any wait.
template <int CH>
__device__ __forceinline__ void router_tile(const RouterArgs& a, uint4* xs, int* status) {
  __shared__ float red[kRouterWarps][kRouterTokens];
  __shared__ __align__(8) uint64_t xbar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, nch = d >> 3;
  const int rows = a.E + (a.w_sg ? 1 : 0);
  const int t0 = blockIdx.y * kRouterTokens;
  const int nt = min(kRouterTokens, a.T - t0);
  const int epc = kRouterWarps / a.wpe;
  const int e = blockIdx.x * epc + warp / a.wpe;
  const int q = warp % a.wpe;

  // Router and gate weights are inputs that no kernel of this library writes:
  // request them before waiting on the predecessor.
  const uint16_t* rowp = (e < a.E) ? a.wr + (size_t)e * d : a.w_sg;
  uint4 w[CH];
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int c = q * 32 + lane + i * a.wpe * 32;
    w[i] = (e < rows && c < nch) ? __ldg(reinterpret_cast<const uint4*>(rowp) + c)
                                 : make_uint4(0, 0, 0, 0);
  }
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
    bulk_g2s(xs, a.x + (size_t)t0 * d, bytes, &xbar, policy_evict_last());
  }
  mbar_wait(&xbar, 0, status);  // on a timeout the logits are garbage; the status says so

  float acc[kRouterTokens];
#pragma unroll
  for (int j = 0; j < kRouterTokens; ++j) {
    acc[j] = 0.f;
    if (j < nt) {
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int c = q * 32 + lane + i * a.wpe * 32;
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
    if (eo < rows && j < nt) {
      float s = 0.f;
      for (int p = 0; p < a.wpe; ++p) s += red[g * a.wpe + p][j];
      if (eo < a.E)
        a.logits[(size_t)(t0 + j) * a.E + eo] = s;
      else
        a.sg[t0 + j] = s;
    }
  }
}

template <int CH>
__global__ void __launch_bounds__(kRouterThreads) router_logits_kernel(RouterArgs a, int* status) {
  extern __shared__ __align__(16) uint4 xs[];
  router_tile<CH>(a, xs, status);
  pdl_trigger();
}

// ------------------------------------------------------------------ top-k
// One warp selects the top-k of one token's E (<= 1024) logits.  Order: larger
// logit first, equal logits -> lower id (softmax is increasing, so this is the
// order of the probabilities).  Weights: exp(l - max) normalised over the
// selected experts (renormalize) or over all E.  Logits are read at L2 (they
// may have been written by other CTAs of the same launch).
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
      v[i] = __ldcg(L + e);
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

// Dispatch on the number of logits each lane holds (E / 32 rounded up to a
// power of two).  Lane j < k receives the j-th selected expert and its weight.
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

// Top-k of token t, stored (lanes j < k) to the routing buffers.
__device__ __forceinline__ void topk_token(const float* logits, int t, int E, int k,
                                           int renormalize, int32_t* ids, float* w,
                                           int32_t* ids_copy, float* w_copy) {
  int id;
  float wt;
  warp_topk(logits + (size_t)t * E, E, k, renormalize, id, wt);
  const int lane = threadIdx.x & 31;
  if (lane < k) {
    const size_t o = (size_t)t * k + lane;
    ids[o] = id;
    w[o] = wt;
    if (ids_copy) ids_copy[o] = id;
    if (w_copy) w_copy[o] = wt;
  }
}

__global__ void __launch_bounds__(256)
    topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renormalize,
                int32_t* ids, float* w, int32_t* ids_copy, float* w_copy) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t < T) topk_token(logits, t, E, k, renormalize, ids, w, ids_copy, w_copy);
}

// ------------------------------------------------------------------ block scan
// Exclusive scan of V ints per thread over the CTA (blockDim a multiple of 32,
// <= 1024).  scratch: >= 32 * V ints.  Every thread gets the totals.
template <int V>
__device__ void block_scan(const int (&v)[V], int (&ex)[V], int (&tot)[V], int* scratch) {
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

// Thread-owned runs of experts: thread i owns [i * run, min(E, (i + 1) * run)).
__device__ __forceinline__ int expert_run(int E) { return (E + blockDim.x - 1) / blockDim.x; }

// ------------------------------------------------------------------ plan
// Estimated cost of a unit with nt tokens, in token-equivalents: a fixed part
// for streaming the unit's weight rows plus one per token of arithmetic.
constexpr int kUnitBaseCost = 4;

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
  // CTA c's share starts at cost c * total / grid, taken in fp32: monotone in c
  // and exact enough for balancing.
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

// Work plan from per-expert counts (cnt) and padded offsets (off), both in
// shared memory: one WorkExpert per touched routed expert (ascending id), then
// the shared expert; unit counts and costs per expert; each CTA's unit range
// for both expert stages.  All threads call it.  tmp: >= 7 * (E + 1) ints.
__device__ void build_plan(const int* cnt, const int* off, int E, int T, int num_post_pad,
                           const PlanParams& pp, int* scratch, int* tmp) {
  const int run = expert_run(E);
  const int e0 = threadIdx.x * run, e1 = min(E, e0 + run);
  // Per-expert values: touched flag, gate_up units, down units, their costs.
  int loc[5] = {0, 0, 0, 0, 0};
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    if (c > 0) {
      const int ggu = (c + pp.xt_gu - 1) / pp.xt_gu, gdn = (c + pp.xt_dn - 1) / pp.xt_dn;
      loc[0] += 1;
      loc[1] += pp.tiles_gu * ggu;
      loc[2] += pp.tiles_dn * gdn;
      loc[3] += pp.tiles_gu * (ggu * kUnitBaseCost + c);
      loc[4] += pp.tiles_dn * (gdn * kUnitBaseCost + c);
    }
  }
  int ex[5], tot[5];
  block_scan<5>(loc, ex, tot, scratch);
  const int W = E + 1;
  int* s_ugu = tmp;
  int* s_udn = tmp + W;
  int* s_cgu = tmp + 2 * W;
  int* s_cdn = tmp + 3 * W;
  int* s_n = tmp + 4 * W;
  int* s_tgu = tmp + 5 * W;
  int* s_tdn = tmp + 6 * W;
  int idx = ex[0], ugu = ex[1], udn = ex[2], cgu = ex[3], cdn = ex[4];
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    if (c == 0) continue;
    const int ggu = (c + pp.xt_gu - 1) / pp.xt_gu, gdn = (c + pp.xt_dn - 1) / pp.xt_dn;
    WorkExpert we;
    we.expert = e;
    we.n_tok = c;
    we.pos = off[e];
    we.unit_gu = ugu;
    we.unit_dn = udn;
    we.pad_[0] = we.pad_[1] = we.pad_[2] = 0;
    pp.work[idx] = we;
    s_ugu[idx] = ugu;
    s_udn[idx] = udn;
    s_cgu[idx] = cgu;
    s_cdn[idx] = cdn;
    s_n[idx] = c;
    s_tgu[idx] = pp.tiles_gu;
    s_tdn[idx] = pp.tiles_dn;
    ++idx;
    ugu += pp.tiles_gu * ggu;
    udn += pp.tiles_dn * gdn;
    cgu += pp.tiles_gu * (ggu * kUnitBaseCost + c);
    cdn += pp.tiles_dn * (gdn * kUnitBaseCost + c);
  }
  const int n_routed = tot[0];
  int tot_gu = tot[1], tot_dn = tot[2], cost_gu = tot[3], cost_dn = tot[4];
  const bool has_shared = pp.tiles_gu_shared > 0 && T > 0;
  const int n_work = n_routed + (has_shared ? 1 : 0);
  if (has_shared) {
    const int sg = (T + pp.xt_gu - 1) / pp.xt_gu, sd = (T + pp.xt_dn - 1) / pp.xt_dn;
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
  split_by_cost(n_work, s_cgu, s_ugu, s_n, s_tgu, cost_gu, tot_gu, pp.xt_gu, pp.grid, pp.cta_gu);
  split_by_cost(n_work, s_cdn, s_udn, s_n, s_tdn, cost_dn, tot_dn, pp.xt_dn, pp.grid, pp.cta_dn);
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

// ------------------------------------------------------------------ align
struct AlignOut {
  int32_t* sorted_ids;
  int32_t* block_ids;
  int32_t* num_post_pad;
  int32_t* expert_offsets;
};

// Shared-memory ints the align step needs for E experts and nw warps; the last
// kAlignSmemSlots hold the routing ids when they fit.
__host__ __device__ constexpr size_t align_smem_ints(int E, int nw) {
  return (size_t)nw * E + 2 * (size_t)E + kScanScratch + 7 * ((size_t)E + 1) + kAlignSmemSlots;
}

// moe_align_block_size (+ the work plan when pp.work) on all threads of the
// CTA.  src: the S = T * k expert ids (shared or global memory).  smem: at
// least align_smem_ints(E, blockDim / 32) ints.
__device__ void align_block(const int32_t* src, int T, int k, int E, int B, const AlignOut& o,
                            const PlanParams& pp, int* status, int* smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int S = T * k;
  int* hist = smem;                   // [nw][E]
  int* cnt = hist + nw * E;           // [E]
  int* off = cnt + E;                 // [E]
  int* scratch = off + E;             // [kScanScratch]
  int* tmp = scratch + kScanScratch;  // [7 * (E + 1)]
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();

  // Phase 1: each warp counts the experts of a contiguous chunk of slots.
  const int chunk = (S + nw - 1) / nw;
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

  // Phase 2: per expert, each warp's exclusive base and the count; padded
  // offsets by a block scan over thread-owned runs of experts.
  const int run = expert_run(E);
  const int e0 = threadIdx.x * run, e1 = min(E, e0 + run);
  int loc[1] = {0};
  for (int e = e0; e < e1; ++e) {
    int r = 0;
    for (int q = 0; q < nw; ++q) {
      const int c = hist[q * E + e];
      hist[q * E + e] = r;
      r += c;
    }
    cnt[e] = r;
    loc[0] += (r + B - 1) / B * B;
  }
  int ex[1], tot[1];
  block_scan<1>(loc, ex, tot, scratch);
  int p0 = ex[0];
  for (int e = e0; e < e1; ++e) {
    const int padded = (cnt[e] + B - 1) / B * B;
    off[e] = p0;
    o.expert_offsets[e] = p0;
    // Pad positions get the sentinel S; every block of the run names e.
    for (int p = p0 + cnt[e]; p < p0 + padded; ++p) o.sorted_ids[p] = S;
    for (int b = p0 / B; b < (p0 + padded) / B; ++b) o.block_ids[b] = e;
    p0 += padded;
  }
  const int total = tot[0];
  if (threadIdx.x == 0) {
    o.expert_offsets[E] = total;
    *o.num_post_pad = total;
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
      o.sorted_ids[off[e] + rank_base + rank] = s;
      if (lane == __ffs(peers) - 1) hist[warp * E + e] = rank_base + __popc(peers);
    }
    __syncwarp();
  }
  if (pp.work != nullptr) build_plan(cnt, off, E, T, total, pp, scratch, tmp);
}

// One CTA of 1024 threads: optional top-k for all T tokens, then align_block.
__global__ void __launch_bounds__(kAlignThreads)
    align_kernel(const float* __restrict__ logits, int T, int E, int k, int renormalize,
                 int32_t* ids, float* w, int32_t* ids_copy, float* w_copy, int B, AlignOut o,
                 PlanParams pp, int* status) {
  extern __shared__ int sm[];
  const int nw = kAlignThreads / 32;
  int* sids = sm + align_smem_ints(E, nw) - kAlignSmemSlots;
  const int S = T * k;
  pdl_wait();
  pdl_trigger();
  if (logits != nullptr) {
    for (int t = threadIdx.x >> 5; t < T; t += nw)
      topk_token(logits, t, E, k, renormalize, ids, w, ids_copy, w_copy);
    __threadfence_block();
    __syncthreads();
  }
  const int32_t* src = ids;
  if (S <= kAlignSmemSlots) {
    for (int s = threadIdx.x; s < S; s += blockDim.x) sids[s] = __ldcg(ids + s);
    src = sids;
  }
  __syncthreads();
  align_block(src, T, k, E, B, o, pp, status, sm);
}

// Plan from an existing align layout (moe_expert_forward): counts recovered
// from the padded runs (a run's trailing sentinel entries are padding).
__global__ void __launch_bounds__(kAlignThreads)
    plan_kernel(int T, int E, int k, int B, const int32_t* __restrict__ sorted_ids,
                const int32_t* __restrict__ num_post_pad, const int32_t* __restrict__ expert_offsets,
                PlanParams pp, int* status) {
  extern __shared__ int sm[];
  int* cnt = sm;                      // [E]
  int* off = cnt + E;                 // [E]
  int* scratch = off + E;             // [kScanScratch]
  int* tmp = scratch + kScanScratch;  // [7 * (E + 1)]
  pdl_wait();
  pdl_trigger();
  const int S = T * k;
  const int cap = S + E * (B - 1);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int o = expert_offsets[e], o1 = expert_offsets[e + 1];
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

// ------------------------------------------------------------------ fused route
struct RouteArgs {
  RouterArgs r;
  int k, renormalize, B;
  int32_t* ids;          // workspace routing [T][k]
  float* w;
  int32_t* ids_copy;     // caller copies (may be null)
  float* w_copy;
  AlignOut o;
  PlanParams pp;
  int* status;
  int* counters;         // [0]: tiles done; [1 + y]: CTAs done in token tile y
};

// Decode-size routing in one launch.  grid = (router CTAs per tile, token
// tiles), 256 threads.  Dynamic shared memory: max(router tile, align step).
// Every CTA arrives on its tile's counter exactly once, whatever happened
// before, so the counters return to zero by the end of every launch.
template <int CH>
__global__ void __launch_bounds__(kRouterThreads) route_kernel(RouteArgs a) {
  extern __shared__ __align__(16) int dsm[];
  __shared__ int s_last;
  router_tile<CH>(a.r, reinterpret_cast<uint4*>(dsm), a.status);
  pdl_trigger();

  // Arrival on this token tile; the last CTA to arrive selects its top-k.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&a.counters[1 + blockIdx.y], 1);
    s_last = old == (int)gridDim.x - 1;
    if (s_last) a.counters[1 + blockIdx.y] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int t = blockIdx.y * kRouterTokens + (threadIdx.x >> 5);
  if ((threadIdx.x >> 5) < kRouterTokens && t < a.r.T)
    topk_token(a.r.logits, t, a.r.E, a.k, a.renormalize, a.ids, a.w, a.ids_copy, a.w_copy);

  // Arrival of this tile; the last tile to finish runs the align and the plan.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&a.counters[0], 1);
    s_last = old == (int)gridDim.y - 1;
    if (s_last) a.counters[0] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int S = a.r.T * a.k;
  int* sids = dsm + align_smem_ints(a.r.E, kRouterWarps) - kAlignSmemSlots;
  for (int s = threadIdx.x; s < S; s += blockDim.x) sids[s] = __ldcg(a.ids + s);
  __syncthreads();
  align_block(sids, a.r.T, a.k, a.r.E, a.B, a.o, a.pp, a.status, dsm);
}

// Router CTA shape: warps per expert row (wpe) and 16-byte chunks per lane.
void router_shape(int T, int d, int rows, int sms, int* wpe_out, int* ch_out) {
  const int ty = (int)ceil_div(T, kRouterTokens);
  const int nch = d / 8;
  int wpe = 8;
  for (int cand = 1; cand <= 8; cand <<= 1) {
    if (ceil_div(rows, kRouterWarps / cand) * ty >= sms) {
      wpe = cand;
      break;
    }
  }
  while (wpe < 8 && ceil_div(nch, wpe * 32) > 8) wpe <<= 1;  // at most 8 chunks per lane
  *wpe_out = wpe;
  *ch_out = (int)ceil_div(nch, wpe * 32);
}

}  // namespace

bool fused_route_supported(int T, int E, int k) {
  return T <= kFusedRouteMaxT && (size_t)T * k <= (size_t)kAlignSmemSlots && E <= 1024;
}

cudaError_t launch_router_logits(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                                 const uint16_t* w_sg, float* logits, float* sg, int T, int d,
                                 int E, int sms, int* status) {
  if (T == 0) return cudaSuccess;
  RouterArgs a{x, wr, w_sg, logits, sg, T, d, E, 0};
  const int rows = E + (w_sg ? 1 : 0);
  int ch;
  router_shape(T, d, rows, sms, &a.wpe, &ch);
  const size_t smem = (size_t)kRouterTokens * d * 2;
  const void* fn = ch <= 1 ? (const void*)router_logits_kernel<1>
                 : ch <= 2 ? (const void*)router_logits_kernel<2>
                 : ch <= 4 ? (const void*)router_logits_kernel<4>
                           : (const void*)router_logits_kernel<8>;
  cudaError_t e = ensure_smem(fn, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(rows, kRouterWarps / a.wpe), (unsigned)ceil_div(T, kRouterTokens));
  void* args[] = {&a, &status};
  return launch_kernel(c, fn, grid, dim3(kRouterThreads), smem, args);
}

cudaError_t launch_route_fused(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                               const uint16_t* w_sg, float* logits, float* sg, int T, int d,
                               int E, int k, int renormalize, int32_t* ids, float* w,
                               int32_t* ids_copy, float* w_copy, int B, int32_t* sorted_ids,
                               int32_t* block_ids, int32_t* num_post_pad, int32_t* expert_offsets,
                               const PlanParams& pp, int* status, int* counters, int sms) {
  if (T == 0) return cudaSuccess;
  RouteArgs a;
  a.r = RouterArgs{x, wr, w_sg, logits, sg, T, d, E, 0};
  const int rows = E + (w_sg ? 1 : 0);
  int ch;
  router_shape(T, d, rows, sms, &a.r.wpe, &ch);
  a.k = k;
  a.renormalize = renormalize;
  a.B = B;
  a.ids = ids;
  a.w = w;
  a.ids_copy = ids_copy;
  a.w_copy = w_copy;
  a.o = AlignOut{sorted_ids, block_ids, num_post_pad, expert_offsets};
  a.pp = pp;
  a.status = status;
  a.counters = counters;
  size_t smem = (size_t)kRouterTokens * d * 2;
  const size_t asmem = align_smem_ints(E, kRouterWarps) * sizeof(int);
  if (asmem > smem) smem = asmem;
  const void* fn = ch <= 1 ? (const void*)route_kernel<1>
                 : ch <= 2 ? (const void*)route_kernel<2>
                 : ch <= 4 ? (const void*)route_kernel<4>
                           : (const void*)route_kernel<8>;
  cudaError_t e = ensure_smem(fn, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(rows, kRouterWarps / a.r.wpe),
            (unsigned)ceil_div(T, kRouterTokens));
  void* args[] = {&a};
  return launch_kernel(c, fn, grid, dim3(kRouterThreads), smem, args);
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
  const size_t smem = align_smem_ints(E, kAlignThreads / 32) * sizeof(int);
  cudaError_t e = ensure_smem((const void*)align_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  AlignOut o{sorted_ids, block_ids, num_post_pad, expert_offsets};
  PlanParams p = pp;
  void* args[] = {&logits, &T, &E, &k, &renormalize, &ids, &w, &ids_copy, &w_copy, &B,
                  &o, &p, &status};
  return launch_kernel(c, (const void*)align_kernel, dim3(1), dim3(kAlignThreads), smem, args);
}

cudaError_t launch_plan(const LaunchCfg& c, int T, int E, int k, int B,
                        const int32_t* sorted_ids, const int32_t* num_post_pad,
                        const int32_t* expert_offsets, const PlanParams& pp, int* status) {
  const size_t smem = (2 * (size_t)E + kScanScratch + 7 * ((size_t)E + 1)) * sizeof(int);
  cudaError_t e = ensure_smem((const void*)plan_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  PlanParams p = pp;
  void* args[] = {&T, &E, &k, &B, &sorted_ids, &num_post_pad, &expert_offsets, &p, &status};
  return launch_kernel(c, (const void*)plan_kernel, dim3(1), dim3(kAlignThreads), smem, args);
}

}  // namespace moe
