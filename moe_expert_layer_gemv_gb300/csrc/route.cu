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
// arrival counter) selects that tile's top-k.  The align and the work plan are
// then built by the expert stages themselves, in every CTA's shared memory
// from the routing ids (expert_gemv.cu), or -- when their shared memory cannot
// hold that plan -- by the last token tile of this kernel ("veloGB10", Kernel
// work: the expert routing folded into its neighbours).
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
  int T, d, E, wpe;        // wpe: warps per router row (1, 2, 4 or 8)
};

// Fixed reduction tree of every router logit (and of the shared-expert gate
// logit x . w_sg, which rides as row E): kRouterSplit partial sums per row,
// partial p summing -- one fp32 fma chain per lane, in ascending i -- the
// 16-byte chunks c = 32 p + lane + 32 kRouterSplit i of the row, then a warp
// butterfly over the lanes; the row's value is the partials added in ascending
// p.  A CTA spreads its rows x partials over its warps in any proportion (wpe
// warps per row, kRouterSplit / wpe partials per warp), so the launch shape
// may follow T while every token's arithmetic stays the same: the routing of a
// token does not depend on the other tokens of the call.
constexpr int kRouterSplit = 8;

// Bytes of dynamic shared memory one router CTA stages: its rows, then the
// 8-token tile.
__host__ __device__ constexpr size_t router_smem_bytes(int d, int wpe) {
  return ((size_t)(kRouterWarps / wpe) + kRouterTokens) * d * 2;
}

// Requests this CTA's router rows (rows [blockIdx.x * epc, +epc), index E =
// the gate row) into `wsm` by bulk copy, completing on `bar`.  The router and
// gate weights are inputs no kernel of this library writes, so this may run
// before the dependency wait.
__device__ __forceinline__ void router_rows_request(const RouterArgs& a, uint8_t* wsm,
                                                    uint64_t* bar) {
  const int epc = kRouterWarps / a.wpe;
  const int rows = a.E + (a.w_sg ? 1 : 0);
  const int e0 = blockIdx.x * epc;
  const int n = min(epc, rows - e0);
  const int nr = min(n, a.E - e0);  // routed rows among them
  const uint32_t rb = (uint32_t)a.d * 2;
  uint32_t bytes = (nr > 0 ? (uint32_t)nr * rb : 0u) + (n > nr ? rb : 0u);
  mbar_arrive_expect_tx(bar, bytes);
  const uint64_t pol = policy_evict_first();
  if (nr > 0) bulk_g2s(wsm, a.wr + (size_t)e0 * a.d, nr * rb, bar, pol);
  if (n > nr) bulk_g2s(wsm + (size_t)(nr > 0 ? nr : 0) * rb, a.w_sg, rb, bar, pol);
}

// One router CTA: rows [blockIdx.x * epc, +epc) for one token tile of 8
// tokens.  smem: >= router_smem_bytes(d, wpe), 16-byte aligned.
__device__ __forceinline__ void router_tile(const RouterArgs& a, uint8_t* smem, int* status) {
  __shared__ float red[kRouterWarps][kRouterSplit][kRouterTokens];
  __shared__ __align__(8) uint64_t bars[2];  // [0] router rows, [1] token tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, nch = d >> 3;
  const int epc = kRouterWarps / a.wpe;
  const int rows = a.E + (a.w_sg ? 1 : 0);
  const int t0 = blockIdx.y * kRouterTokens;
  const int nt = min(kRouterTokens, a.T - t0);
  uint8_t* wsm = smem;
  uint8_t* xsm = smem + (size_t)epc * d * 2;

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
    router_rows_request(a, wsm, &bars[0]);
  }
  __syncthreads();
  pdl_wait();
  // The token tile is contiguous: one bulk copy.
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)nt * d * 2;
    mbar_arrive_expect_tx(&bars[1], bytes);
    bulk_g2s(xsm, a.x + (size_t)t0 * d, bytes, &bars[1], policy_evict_last());
  }
  // On a timeout the logits are garbage; the status word says so.
  mbar_wait(&bars[0], 0, status);
  mbar_wait(&bars[1], 0, status);

  const int r = warp / a.wpe;                 // row of this CTA
  const int G = kRouterSplit / a.wpe;         // partials of this warp
  const int p0 = (warp % a.wpe) * G;
  const bool live = blockIdx.x * epc + r < rows;
  const uint32_t wrow = smem_u32(wsm) + (uint32_t)(r * d * 2);
  const uint32_t xrow = smem_u32(xsm);
  for (int g = 0; g < G && live; ++g) {
    const int p = p0 + g;
    float acc[kRouterTokens];
#pragma unroll
    for (int j = 0; j < kRouterTokens; ++j) acc[j] = 0.f;
    for (int c = 32 * p + lane; c < nch; c += 32 * kRouterSplit) {
      uint4 wv;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(wv.x), "=r"(wv.y), "=r"(wv.z), "=r"(wv.w)
                   : "r"(wrow + c * 16));
#pragma unroll
      for (int j = 0; j < kRouterTokens; ++j) {
        if (j < nt) {
          uint4 xv;
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                       : "r"(xrow + (uint32_t)(j * d * 2 + c * 16)));
          acc[j] = dot8_bf16(wv, xv, acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kRouterTokens; ++j) acc[j] = warp_sum(acc[j]);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kRouterTokens; ++j) red[r][p][j] = acc[j];
    }
  }
  __syncthreads();
  if (threadIdx.x < epc * kRouterTokens) {
    const int g = threadIdx.x / kRouterTokens, j = threadIdx.x % kRouterTokens;
    const int eo = blockIdx.x * epc + g;
    if (eo < rows && j < nt) {
      float v = 0.f;
#pragma unroll
      for (int p = 0; p < kRouterSplit; ++p) v += red[g][p][j];
      if (eo < a.E)
        a.logits[(size_t)(t0 + j) * a.E + eo] = v;
      else
        a.sg[t0 + j] = v;
    }
  }
}

__global__ void __launch_bounds__(kRouterThreads) router_logits_kernel(RouterArgs a, int* status) {
  extern __shared__ __align__(16) uint8_t rsm[];
  router_tile(a, rsm, status);
  pdl_trigger();
}

// ------------------------------------------------------------------ top-k
// One warp selects the top-k of one token's E (<= 1024) logits.  Order: larger
// logit first, equal logits -> lower id (softmax is increasing, so this is the
// order of the probabilities).  Each lane sorts its NV logits (ids lane + 32 i)
// once; then each of the k rounds is one warp max over the lanes' heads and
// one warp min over the ids holding it, and the winning lane pops its head.
// Weights: exp(l - max) normalised over the selected experts (renormalize) or
// over all E.  Logits are read at L2 (they may have been written by other CTAs
// of the same launch).

// Order-preserving map of a float to an unsigned key (key 0 is never produced
// by a finite or infinite float, so it marks an empty slot).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;  // -0 and +0 are the same logit
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NV>
__device__ void warp_topk_nv(const float* __restrict__ L, int E, int k, int renormalize,
                             int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NV];
  int id[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    id[i] = e;
    key[i] = e < E ? float_key(__ldcg(L + e)) : 0u;
  }
  // Per-lane sort, descending key; equal keys keep ascending id (stable).
#pragma unroll
  for (int pass = 0; pass < NV; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < NV; i += 2) {
      if (key[i + 1] > key[i]) {
        const uint32_t tk = key[i];
        key[i] = key[i + 1];
        key[i + 1] = tk;
        const int ti = id[i];
        id[i] = id[i + 1];
        id[i + 1] = ti;
      }
    }
  }
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key[0]);
  const float mx = key_float(kmax);
  float z = 0.f;
  if (!renormalize) {
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (key[i] != 0u) z += expf(key_float(key[i]) - mx);
    z = warp_sum(z);
  }
  int my_id = 0;
  uint32_t my_key = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t win = __reduce_min_sync(0xffffffffu, key[0] == m ? (uint32_t)id[0] : 0xffffffffu);
    if (lane == j) {
      my_id = (int)win;
      my_key = m;
    }
    if (key[0] == m && (uint32_t)id[0] == win) {  // the winning lane pops its head
#pragma unroll
      for (int i = 0; i + 1 < NV; ++i) {
        key[i] = key[i + 1];
        id[i] = id[i + 1];
      }
      key[NV - 1] = 0u;
    }
  }
  const float ev = lane < k ? expf(key_float(my_key) - mx) : 0.f;
  out_id = my_id;
  out_w = ev / (renormalize ? warp_sum(ev) : z);
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

// Top-k of token t, stored (lanes j < k) to the routing buffers (and, when
// ids_smem, to shared memory at the same slot index).  NV > 0: the logits per
// lane are known at compile time (E <= 32 NV); 0: dispatch on E.
template <int NV = 0>
__device__ __forceinline__ void topk_token(const float* logits, int t, int E, int k,
                                           int renormalize, int32_t* ids, float* w,
                                           int32_t* ids_copy, float* w_copy,
                                           int32_t* ids_smem = nullptr) {
  int id;
  float wt;
  if (NV > 0)
    warp_topk_nv<NV ? NV : 1>(logits + (size_t)t * E, E, k, renormalize, id, wt);
  else
    warp_topk(logits + (size_t)t * E, E, k, renormalize, id, wt);
  const int lane = threadIdx.x & 31;
  if (lane < k) {
    const size_t o = (size_t)t * k + lane;
    ids[o] = id;
    w[o] = wt;
    if (ids_smem) ids_smem[o] = id;
    if (ids_copy) ids_copy[o] = id;
    if (w_copy) w_copy[o] = wt;
  }
}

// One warp per token: its top-k and, when sg, the shared-expert gate logit
// sg[t] = x[t] . w_sg (fp32, lane partials then the warp's butterfly sum).
__global__ void __launch_bounds__(256)
    topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renormalize,
                int32_t* ids, float* w, int32_t* ids_copy, float* w_copy,
                const uint16_t* __restrict__ x, int d, const uint16_t* __restrict__ w_sg,
                float* sg) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_token(logits, t, E, k, renormalize, ids, w, ids_copy, w_copy);
  if (sg != nullptr) {
    const int lane = threadIdx.x & 31;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const uint4* gr = reinterpret_cast<const uint4*>(w_sg);
    float acc = 0.f;
    for (int c = lane; c < d / 8; c += 32) acc = dot8_bf16(xr[c], gr[c], acc);
    acc = warp_sum(acc);
    if (lane == 0) sg[t] = acc;
  }
}

// Thread-owned runs of experts: thread i owns [i * run, min(E, (i + 1) * run)).
__device__ __forceinline__ int expert_run(int E) { return (E + blockDim.x - 1) / blockDim.x; }

// ------------------------------------------------------------------ plan
// Estimated cost of a unit with nt tokens, in token-equivalents: a fixed part
// `base` for streaming (and, int4, dequantising) the unit's weight rows plus
// tok_w per token of arithmetic (1 for the shared expert's units).  The routed experts' base and the shared
// expert's are separate (PlanParams::base_gu / base_gu_s, base_dn / base_dn_s).

// CTA c of one stage gets units [cta[c], cta[c+1]) and starts in work expert
// cta[grid + 1 + c]: its share of the stage's estimated cost starts at
// split_target(c) (taken in fp32: monotone in c, exact enough for balancing).
// cta[grid] is where the dynamic tail starts, in work expert cta[2 grid + 1]
// (without a tail: the total of units).
__device__ void split_one(int c, int n_work, const int* s_cost, const int* s_unit, const int* s_n,
                          const int* s_tiles, int total_cost, int xt, int base,
                          int base_s, int tw, bool tile_major, bool has_shared, bool tail,
                          int total_units, int grid, float skew, int32_t* cta) {
  if (n_work == 0) {
    cta[c] = 0;
    cta[grid + 1 + c] = 0;
    return;
  }
  if (c == grid && !tail) {
    cta[c] = total_units;
    cta[2 * grid + 1] = n_work - 1;
    return;
  }
  const int target = split_target(c, grid, total_cost, tail, skew);
  int lo = 0, hi = n_work - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_cost[mid] <= target) lo = mid; else hi = mid - 1;
  }
  const bool sh = has_shared && lo == n_work - 1;
  cta[c] = c == 0 ? 0 : unit_at_cost(target, s_cost[lo], s_unit[lo], s_tiles[lo], s_n[lo], xt,
                                      sh ? base_s : base, sh ? 1 : tw, tile_major);
  cta[grid + 1 + c] = lo;
}

// Per-expert quantities scanned over the experts: padded length, touched
// flag, gate_up units, down units, their estimated costs, and (tensor-core
// path) gate_up and down tiles of 128 rows.
constexpr int kVals = 8;
constexpr int kTcRows = 128;
__device__ __forceinline__ void expert_vals(int c, int B, const PlanParams& pp, int (&v)[kVals]) {
  const int ggu = (c + pp.xt_gu - 1) / pp.xt_gu, gdn = (c + pp.xt_dn - 1) / pp.xt_dn;
  const int mb = (c + kTcRows - 1) / kTcRows;
  const bool t = c > 0;
  v[0] = (c + B - 1) / B * B;
  v[1] = t ? 1 : 0;
  v[2] = t ? pp.tiles_gu * ggu : 0;
  v[3] = t ? pp.tiles_dn * gdn : 0;
  v[4] = t ? pp.tiles_gu * (ggu * pp.base_gu + pp.tok_w * c) : 0;
  v[5] = t ? pp.tiles_dn * (gdn * pp.base_dn + pp.tok_w * c) : 0;
  v[6] = mb * pp.tc_nb_gu;
  v[7] = mb * pp.tc_nb_dn;
}

struct AlignOut {
  int32_t* sorted_ids;
  int32_t* block_ids;
  int32_t* num_post_pad;
  int32_t* expert_offsets;
};

// Plan totals every thread needs for the split.
struct PlanTotals {
  int n_work, units_gu, units_dn, cost_gu, cost_dn, num_post_pad, tc_gu, tc_dn;
  bool has_shared;  // the last work expert is the shared expert
};

// From per-expert counts cnt[E] (shared memory): one block scan of the
// expert_vals over thread-owned runs of experts, then
//   - when o: padded offsets into off[] and the align outputs (offsets,
//     sentinel pads, block ids, num_post_pad); otherwise off[] is given;
//   - when pp.work: the work list (one entry per touched expert, ascending id,
//     then the shared expert) and the arrays split_stages() searches.
// Ends with a CTA barrier.  tmp: >= 7 * (E + 1) ints; scratch: kScanScratch.
__device__ PlanTotals layout_and_plan(const int* cnt, int* off, int E, int T, int S, int B,
                                      const AlignOut* o, const PlanParams& pp, int* scratch,
                                      int* tmp) {
  const int run = expert_run(E);
  const int e0 = threadIdx.x * run, e1 = min(E, e0 + run);
  int loc[kVals] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int e = e0; e < e1; ++e) {
    int v[kVals];
    expert_vals(cnt[e], B, pp, v);
#pragma unroll
    for (int i = 0; i < kVals; ++i) loc[i] += v[i];
  }
  int ex[kVals], tot[kVals];
  block_scan<kVals>(loc, ex, tot, scratch);
  const int W = E + 1;
  int* s_ugu = tmp;
  int* s_udn = tmp + W;
  int* s_cgu = tmp + 2 * W;
  int* s_cdn = tmp + 3 * W;
  int* s_n = tmp + 4 * W;
  int* s_tgu = tmp + 5 * W;
  int* s_tdn = tmp + 6 * W;
  int acc[kVals];
#pragma unroll
  for (int i = 0; i < kVals; ++i) acc[i] = ex[i];
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    int v[kVals];
    expert_vals(c, B, pp, v);
    if (o != nullptr) {
      const int p0 = acc[0];
      off[e] = p0;
      o->expert_offsets[e] = p0;
      // Pad positions get the sentinel S; every block of the run names e.
      for (int p = p0 + c; p < p0 + v[0]; ++p) o->sorted_ids[p] = S;
      for (int b = p0 / B; b < (p0 + v[0]) / B; ++b) o->block_ids[b] = e;
    }
    if (pp.work != nullptr && c > 0) {
      const int idx = acc[1];
      WorkExpert we;
      we.expert = e;
      we.n_tok = c;
      we.pos = off[e];
      we.unit_gu = acc[2];
      we.unit_dn = acc[3];
      we.pad_[0] = acc[6];  // first tensor-core tile, gate_up
      we.pad_[1] = acc[7];  // first tensor-core tile, down
      we.pad_[2] = 0;
      pp.work[idx] = we;
      s_ugu[idx] = acc[2];
      s_udn[idx] = acc[3];
      s_cgu[idx] = acc[4];
      s_cdn[idx] = acc[5];
      s_n[idx] = c;
      s_tgu[idx] = pp.tiles_gu;
      s_tdn[idx] = pp.tiles_dn;
    }
#pragma unroll
    for (int i = 0; i < kVals; ++i) acc[i] += v[i];
  }
  if (o != nullptr && threadIdx.x == 0) {
    o->expert_offsets[E] = tot[0];
    *o->num_post_pad = tot[0];
  }
  PlanTotals pt{tot[1], tot[2], tot[3], tot[4], tot[5], tot[0], tot[6], tot[7], false};
  if (pp.work != nullptr && pp.tiles_gu_shared > 0 && T > 0) {
    const int sg = (T + pp.xt_gu - 1) / pp.xt_gu, sd = (T + pp.xt_dn - 1) / pp.xt_dn;
    if (threadIdx.x == 0) {
      WorkExpert we;
      we.expert = -1;
      we.n_tok = T;
      we.pos = 0;
      we.unit_gu = pt.units_gu;
      we.unit_dn = pt.units_dn;
      we.pad_[0] = pt.tc_gu;
      we.pad_[1] = pt.tc_dn;
      we.pad_[2] = 0;
      pp.work[pt.n_work] = we;
      s_ugu[pt.n_work] = pt.units_gu;
      s_udn[pt.n_work] = pt.units_dn;
      s_cgu[pt.n_work] = pt.cost_gu;
      s_cdn[pt.n_work] = pt.cost_dn;
      s_n[pt.n_work] = T;
      s_tgu[pt.n_work] = pp.tiles_gu_shared;
      s_tdn[pt.n_work] = pp.tiles_dn_shared;
    }
    pt.n_work += 1;
    pt.has_shared = true;
    pt.units_gu += pp.tiles_gu_shared * sg;
    pt.units_dn += pp.tiles_dn_shared * sd;
    pt.cost_gu += pp.tiles_gu_shared * (sg * pp.base_gu_s + T);
    pt.cost_dn += pp.tiles_dn_shared * (sd * pp.base_dn_s + T);
    const int mbs = (T + kTcRows - 1) / kTcRows;
    pt.tc_gu += mbs * pp.tc_nb_gu;
    pt.tc_dn += mbs * pp.tc_nb_dn;
  }
  __syncthreads();
  return pt;
}

// Both stages' CTA ranges (one pass over 2 * (grid + 1) items) and the Plan.
__device__ void split_stages(const PlanTotals& pt, int E, const PlanParams& pp, const int* tmp) {
  const int W = E + 1;
  const int per = pp.grid + 1;
  // The tensor-core kernels walk the plan by tiles, not by these ranges.
  for (int i = threadIdx.x; pp.tc_nb_gu == 0 && i < 2 * per; i += blockDim.x) {
    if (i < per)
      split_one(i, pt.n_work, tmp + 2 * W, tmp, tmp + 4 * W, tmp + 5 * W, pt.cost_gu, pp.xt_gu,
                pp.base_gu, pp.base_gu_s, pp.tok_w, pp.tile_major != 0, pt.has_shared,
                pp.tail_gu != 0, pt.units_gu,
                pp.grid, 0.f, pp.cta_gu);
    else
      split_one(i - per, pt.n_work, tmp + 3 * W, tmp + W, tmp + 4 * W, tmp + 6 * W, pt.cost_dn,
                pp.xt_dn, pp.base_dn, pp.base_dn_s, pp.tok_w, pp.tile_major != 0, pt.has_shared,
                pp.tail_dn != 0,
                pt.units_dn, pp.grid, pp.tail_dn ? 0.f : kDownSkew, pp.cta_dn);
  }
  if (threadIdx.x == 0) {
    Plan p;
    p.n_work = pt.n_work;
    p.units_gu = pt.units_gu;
    p.units_dn = pt.units_dn;
    p.num_post_pad = pt.num_post_pad;
    p.pad_[0] = pt.tc_gu;  // tensor-core tiles, gate_up
    p.pad_[1] = pt.tc_dn;  // tensor-core tiles, down
    p.pad_[2] = p.pad_[3] = 0;
    *pp.plan = p;
  }
}

// ------------------------------------------------------------------ align
// Shared-memory ints the single-CTA align needs for E experts; the last
// kAlignSmemSlots hold the routing ids, the ones before them their ranks.
__host__ __device__ constexpr size_t align_smem_ints(int E) {
  return 2 * (size_t)E + kScanScratch + 7 * ((size_t)E + 1) + 2 * (size_t)kAlignSmemSlots;
}

// moe_align_block_size (+ the work plan when pp.work) on all threads of one
// CTA, for S <= kAlignSmemSlots with the ids in shared memory (sids): warp 0
// walks the slots in order, 32 at a time, giving every slot its rank among the
// earlier slots of its expert.
__device__ void align_block_small(const int32_t* sids, int T, int k, int E, int B,
                                  const AlignOut& o, const PlanParams& pp, int* status,
                                  int* smem) {
  const int lane = threadIdx.x & 31;
  const int S = T * k;
  int* cnt = smem;                    // [E]
  int* off = cnt + E;                 // [E]
  int* scratch = off + E;             // [kScanScratch]
  int* tmp = scratch + kScanScratch;  // [7 * (E + 1)]
  int* rank = tmp + 7 * (E + 1);      // [S]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    for (int base = 0; base < S; base += 32) {
      const int s = base + lane;
      int e = -1;
      if (s < S) {
        e = sids[s];
        if (e < 0 || e >= E) {
          record_status(status, kStatusDeviceCheck);
          e = -1;
        }
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) rank[s] = cnt[e] + __popc(peers & ((1u << lane) - 1u));
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  const PlanTotals pt = layout_and_plan(cnt, off, E, T, S, B, &o, pp, scratch, tmp);
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int e = sids[s];
    if (e >= 0 && e < E) o.sorted_ids[off[e] + rank[s]] = s;
  }
  if (pp.work != nullptr) split_stages(pt, E, pp, tmp);
}

// One CTA of 1024 threads: the align (and plan) of S <= kAlignSmemSlots
// routing ids.
__global__ void __launch_bounds__(kAlignThreads)
    align_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int B, AlignOut o,
                 PlanParams pp, int* status) {
  extern __shared__ int sm[];
  int* sids = sm + align_smem_ints(E) - kAlignSmemSlots;
  const int S = T * k;
  pdl_wait();
  pdl_trigger();
  for (int s = threadIdx.x; s < S; s += blockDim.x) sids[s] = __ldcg(ids + s);
  __syncthreads();
  align_block_small(sids, T, k, E, B, o, pp, status, sm);
}

// Larger S: chunks of kAlignThreads slots, one per CTA of align_count_kernel.
// Each CTA ranks its slots among the earlier slots of the chunk with the same
// expert (match within a warp, per-warp histograms across warps) and stores
// the chunk's count of every expert; the last CTA to finish turns the counts
// into per-chunk bases (a scan over the chunks of each expert, one warp per
// expert), lays out the padded runs and builds the plan.  align_emit_kernel
// then places every slot at offset[e] + base[e][chunk] + rank: the same
// arrival order as one in-order pass.
struct AlignChunks {
  int32_t* base;     // [E][nch]: count of expert e in chunk c, then its exclusive base
  int32_t* rank;     // [S]
  int* counter;      // CTAs finished (zero between launches)
};

__global__ void __launch_bounds__(kAlignThreads)
    align_count_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int B, AlignOut o,
                       PlanParams pp, AlignChunks ac, int* status) {
  extern __shared__ int sm[];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = kAlignThreads / 32;
  const int S = T * k, nch = gridDim.x, c = blockIdx.x;
  int* whist = sm;  // [nw][E]
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  const int s = c * kAlignThreads + threadIdx.x;
  int e = -1;
  if (s < S) {
    e = __ldcg(ids + s);
    if (e < 0 || e >= E) {
      record_status(status, kStatusDeviceCheck);
      e = -1;
    }
  }
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  if (e >= 0 && lane == __ffs(peers) - 1) whist[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int r = 0;
    for (int q = 0; q < nw; ++q) {
      const int v = whist[q * E + x];
      whist[q * E + x] = r;
      r += v;
    }
    ac.base[(size_t)x * nch + c] = r;
  }
  __syncthreads();
  if (e >= 0) ac.rank[s] = whist[warp * E + e] + __popc(peers & ((1u << lane) - 1u));

  // Arrival; the last CTA sees every chunk's counts.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(ac.counter, 1);
    s_last = old == nch - 1;
    if (s_last) *ac.counter = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int* cnt = sm;                      // [E]
  int* off = cnt + E;                 // [E]
  int* scratch = off + E;             // [kScanScratch]
  int* tmp = scratch + kScanScratch;  // [7 * (E + 1)]
  for (int x = warp; x < E; x += nw) {
    int run = 0;
    for (int c0 = 0; c0 < nch; c0 += 32) {
      const int ch = c0 + lane;
      const int v = ch < nch ? __ldcg(ac.base + (size_t)x * nch + ch) : 0;
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += u;
      }
      if (ch < nch) ac.base[(size_t)x * nch + ch] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) cnt[x] = run;
  }
  __syncthreads();
  const PlanTotals pt = layout_and_plan(cnt, off, E, T, S, B, &o, pp, scratch, tmp);
  if (pp.work != nullptr) split_stages(pt, E, pp, tmp);
}

__global__ void __launch_bounds__(kAlignThreads)
    align_emit_kernel(const int32_t* __restrict__ ids, int T, int E, int k, AlignOut o,
                      AlignChunks ac) {
  pdl_wait();
  pdl_trigger();
  const int S = T * k, nch = gridDim.x, c = blockIdx.x;
  const int s = c * kAlignThreads + threadIdx.x;
  if (s >= S) return;
  const int e = __ldcg(ids + s);
  if (e < 0 || e >= E) return;  // recorded by align_count_kernel
  o.sorted_ids[__ldcg(o.expert_offsets + e) + __ldcg(ac.base + (size_t)e * nch + c) +
               __ldcg(ac.rank + s)] = s;
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
  PlanTotals pt = layout_and_plan(cnt, off, E, T, S, B, nullptr, pp, scratch, tmp);
  pt.num_post_pad = *num_post_pad;
  split_stages(pt, E, pp, tmp);
}

// ------------------------------------------------------------------ fused route
struct RouteArgs {
  RouterArgs r;
  int k, renormalize, B;
  int align;             // 1: the last token tile also runs the align and the plan
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
// NV: logits per lane of the top-k (E <= 32 NV), so that each instantiation
// holds only the registers its E needs (two CTAs per SM).
template <int NV>
__global__ void __launch_bounds__(kRouterThreads, NV >= 32 ? 1 : 2) route_kernel(RouteArgs a) {
  extern __shared__ __align__(16) int dsm[];
  __shared__ int s_last;
  router_tile(a.r, reinterpret_cast<uint8_t*>(dsm), a.status);
  pdl_trigger();

  // Arrival on this token tile; the last CTA to arrive selects its top-k.
  // The barrier orders the CTA's logit stores before thread 0's arrival, whose
  // release publishes them; the last arrival's acquire, passed on by the
  // second barrier, makes every CTA's logits of the tile visible here.
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atom_add_acq_rel_gpu(&a.counters[1 + blockIdx.y], 1);
    s_last = old == (int)gridDim.x - 1;
    if (s_last) a.counters[1 + blockIdx.y] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  const int t = blockIdx.y * kRouterTokens + (threadIdx.x >> 5);
  // With one token tile this CTA runs the align too: the ids go straight to
  // its shared-memory slots (the router's x tile there is no longer needed).
  int* sids = dsm + align_smem_ints(a.r.E) - kAlignSmemSlots;
  if ((threadIdx.x >> 5) < kRouterTokens && t < a.r.T)
    topk_token<NV>(a.r.logits, t, a.r.E, a.k, a.renormalize, a.ids, a.w, a.ids_copy, a.w_copy,
                   gridDim.y == 1 && a.align ? sids : nullptr);
  // Without the align here, the expert stages plan from the ids themselves.
  if (!a.align) return;

  // Arrival of this tile; the last tile to finish runs the align and the plan
  // (with one token tile, this CTA is already the last).
  __threadfence();
  __syncthreads();
  if (gridDim.y > 1) {
    if (threadIdx.x == 0) {
      const int old = atomicAdd(&a.counters[0], 1);
      s_last = old == (int)gridDim.y - 1;
      if (s_last) a.counters[0] = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  if (gridDim.y > 1) {
    const int S = a.r.T * a.k;
    for (int s = threadIdx.x; s < S; s += blockDim.x) sids[s] = __ldcg(a.ids + s);
    __syncthreads();
  }
  align_block_small(sids, a.r.T, a.k, a.r.E, a.B, a.o, a.pp, a.status, dsm);
}

// Router CTA shape: warps per router row.  The arithmetic is the same for
// every shape (kRouterSplit), so the choice only sets the parallelism: the
// fewest CTAs that still cover every SM (each CTA stages the whole token tile,
// so fewer CTAs move fewer bytes), within the shared memory a CTA may hold.
int router_wpe(int T, int d, int rows, int sms) {
  const int ty = (int)ceil_div(T, kRouterTokens);
  for (int wpe = 1; wpe <= 8; wpe <<= 1) {
    if (router_smem_bytes(d, wpe) > 200 * 1024) continue;
    if (wpe == 8 || ceil_div(rows, kRouterWarps / wpe) * ty >= sms) return wpe;
  }
  return 8;
}

size_t route_fused_smem(int d, int E, int wpe) {
  const size_t a = align_smem_ints(E) * sizeof(int);
  const size_t r = router_smem_bytes(d, wpe);
  return a > r ? a : r;
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
  a.wpe = router_wpe(T, d, rows, sms);
  const size_t smem = router_smem_bytes(d, a.wpe);
  const void* fn = (const void*)router_logits_kernel;
  cudaError_t e = ensure_smem(fn, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(rows, kRouterWarps / a.wpe), (unsigned)ceil_div(T, kRouterTokens));
  void* args[] = {&a, &status};
  return launch_kernel(c, fn, grid, dim3(kRouterThreads), smem, args);
}

cudaError_t launch_route_fused(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                               const uint16_t* w_sg, float* logits, float* sg, int T, int d,
                               int E, int k, int renormalize, int32_t* ids, float* w,
                               int32_t* ids_copy, float* w_copy, bool align, int B,
                               int32_t* sorted_ids, int32_t* block_ids, int32_t* num_post_pad,
                               int32_t* expert_offsets, const PlanParams& pp, int* status,
                               int* counters, int sms) {
  if (T == 0) return cudaSuccess;
  RouteArgs a;
  a.r = RouterArgs{x, wr, w_sg, logits, sg, T, d, E, 0};
  const int rows = E + (w_sg ? 1 : 0);
  a.r.wpe = router_wpe(T, d, rows, sms);
  a.k = k;
  a.renormalize = renormalize;
  a.B = B;
  a.align = align ? 1 : 0;
  a.ids = ids;
  a.w = w;
  a.ids_copy = ids_copy;
  a.w_copy = w_copy;
  a.o = AlignOut{sorted_ids, block_ids, num_post_pad, expert_offsets};
  a.pp = pp;
  a.status = status;
  a.counters = counters;
  const size_t smem = align ? route_fused_smem(d, E, a.r.wpe) : router_smem_bytes(d, a.r.wpe);
  const int nv = (E + 31) / 32;
  const void* fn = nv <= 1 ? (const void*)route_kernel<1>
                 : nv <= 2 ? (const void*)route_kernel<2>
                 : nv <= 4 ? (const void*)route_kernel<4>
                 : nv <= 8 ? (const void*)route_kernel<8>
                 : nv <= 16 ? (const void*)route_kernel<16>
                            : (const void*)route_kernel<32>;
  cudaError_t e = ensure_smem(fn, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(rows, kRouterWarps / a.r.wpe),
            (unsigned)ceil_div(T, kRouterTokens));
  void* args[] = {&a};
  return launch_kernel(c, fn, grid, dim3(kRouterThreads), smem, args);
}

cudaError_t launch_topk(const LaunchCfg& c, const float* logits, int T, int E, int k,
                        int renormalize, int32_t* ids, float* w, int32_t* ids_copy,
                        float* w_copy, const uint16_t* x, int d, const uint16_t* w_sg,
                        float* sg) {
  if (T == 0) return cudaSuccess;
  dim3 grid((unsigned)ceil_div(T, 8));
  void* args[] = {&logits, &T, &E, &k, &renormalize, &ids, &w, &ids_copy, &w_copy,
                  &x, &d, &w_sg, &sg};
  return launch_kernel(c, (const void*)topk_kernel, grid, dim3(256), 0, args);
}

int align_chunks(int T, int k) { return (int)ceil_div((int64_t)T * k, kAlignThreads); }

cudaError_t launch_align(const LaunchCfg& c, const int32_t* ids, int T, int E, int k, int B,
                         int32_t* sorted_ids, int32_t* block_ids, int32_t* num_post_pad,
                         int32_t* expert_offsets, const PlanParams& pp, int* status,
                         int32_t* chunk_base, int32_t* chunk_rank, int* counter) {
  AlignOut o{sorted_ids, block_ids, num_post_pad, expert_offsets};
  PlanParams p = pp;
  if ((int64_t)T * k <= kAlignSmemSlots) {
    const size_t smem = align_smem_ints(E) * sizeof(int);
    cudaError_t e = ensure_smem((const void*)align_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {&ids, &T, &E, &k, &B, &o, &p, &status};
    return launch_kernel(c, (const void*)align_kernel, dim3(1), dim3(kAlignThreads), smem, args);
  }
  const int nw = kAlignThreads / 32;
  const size_t need = (size_t)nw * E > 2 * (size_t)E + kScanScratch + 7 * ((size_t)E + 1)
                          ? (size_t)nw * E
                          : 2 * (size_t)E + kScanScratch + 7 * ((size_t)E + 1);
  const size_t smem = need * sizeof(int);
  cudaError_t e = ensure_smem((const void*)align_count_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  AlignChunks ac{chunk_base, chunk_rank, counter};
  const dim3 grid((unsigned)align_chunks(T, k));
  void* args[] = {&ids, &T, &E, &k, &B, &o, &p, &ac, &status};
  if ((e = launch_kernel(c, (const void*)align_count_kernel, grid, dim3(kAlignThreads), smem,
                         args)) != cudaSuccess)
    return e;
  void* eargs[] = {&ids, &T, &E, &k, &o, &ac};
  return launch_kernel(LaunchCfg{c.stream, true}, (const void*)align_emit_kernel, grid,
                       dim3(kAlignThreads), 0, eargs);
}

cudaError_t launch_plan(const LaunchCfg& c, int T, int E, int k, int B,
                        const int32_t* sorted_ids, const int32_t* num_post_pad,
                        const int32_t* expert_offsets, const PlanParams& pp, int* status) {
  const size_t smem = (2 * (size_t)E + kScanScratch + 7 * ((size_t)E + 1)) * sizeof(int);  // plan_kernel
  cudaError_t e = ensure_smem((const void*)plan_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  PlanParams p = pp;
  void* args[] = {&T, &E, &k, &B, &sorted_ids, &num_post_pad, &expert_offsets, &p, &status};
  return launch_kernel(c, (const void*)plan_kernel, dim3(1), dim3(kAlignThreads), smem, args);
}

}  // namespace moe
