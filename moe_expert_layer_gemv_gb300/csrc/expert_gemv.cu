// expert_gemv.cu -- grouped expert GEMVs for small T (decode / speculative
// verify): gate_up + SwiGLU, then down.  Only the touched experts' weights are
// read, each byte once from HBM ("veloGB10", Kernel work: grouped MoE expert
// kernels that never rebuild full weights; shared-expert work overlapped with
// the MoE step -- here the shared expert is one more work expert in the same
// persistent grid).
//
// Structure (both stages): a persistent grid of kCtasPerSm CTAs per SM.  Work
// is cut into units = (work expert, token group, row tile); each CTA takes one
// contiguous range of units of about equal estimated cost (and, on long
// stages, units of the dynamic tail one at a time).  At decode sizes every CTA
// derives the plan (align layout, work list, its range) from the routing ids
// in its own shared memory (smem_plan; one warp for up to 64 slots);
// otherwise it reads the plan the align step wrote to the workspace.  The last
// warp of a CTA is the producer: bulk copies (bf16 weight blocks, activation
// rows) and tiled tensor copies (int4 code boxes, 128-byte swizzle) land a unit
// in a shared-memory ring stage and complete the stage's mbarrier by
// transaction bytes.  The other warps consume, then release the stage:
// - bf16: fp32 dot products out of shared memory (packed fp32 fma, several
//   accumulators per output, warp-shuffle reductions), the token count a
//   template parameter so the inner loops carry no per-token branches;
// - int4: the codes dequantised in registers (two nibbles per bf16 pair, one
//   packed fma) and multiplied on the tensor pipe (mma.sync m16n8k16, bf16,
//   fp32 accumulation), each group's products scaled by its bf16 scale (W4A16
//   routed experts, group size 32: "Qwen3.8 Flash-Next - GB10 UltraFast", How
//   it works; Manual).
// Then the SwiGLU (gate_up) or the per-slot output write (down).
#include <cuda_bf16.h>

#include <cstring>

#include "launch.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxXT = 8;          // tokens per unit
constexpr int kBarBytes = 256;     // barrier area at the start of shared memory
constexpr int kMaxStages = 8;

struct GuArgs {
  CUtensorMap tm_codes;       // int4: codes as {128-byte chunk, row of [E*2I], chunk of d/256},
                              // box {128, 8, d/256}, 128-byte swizzle
  const uint8_t* gu;          // routed gate_up: bf16 [E][2I][d] or codes [E][2I][d/2]
  const uint16_t* gu_scales;  // int4 scales [E][2I][d/32]
  const uint8_t* sgu;         // shared gate_up bf16 [2Is][d] (may be null)
  const uint8_t* sdn;         // shared down bf16 [d][Is] (prefetched into L2 only)
  const uint16_t* x;          // [T][d]
  const int32_t* sorted_ids;
  const Plan* plan;
  const WorkExpert* work;
  const int32_t* cta;         // CTA unit ranges and first work experts (see PlanParams)
  float* h;                   // [sorted positions][I]; int4 layers: two bf16 planes
  float* hs;                  // [T][Is]
  int* status;
  int* dyn;                   // the stage's dynamic-tail ticket counter (DynTail)
  int* dyn_other;             // the down stage's, zeroed here
  int T, d, I, Is, k;
  int rg, rgs, xt, stage_bytes, n_stages;
  int stage_off;              // shared-memory offset of the stage ring
  int h_rows;                 // rows of each bf16 plane of h (int4 layers)
  SmemPlanArgs sp;
};

struct DnArgs {
  CUtensorMap tm_codes;       // int4: codes as [E*d][I/2] bytes, box {128, 64}, 128-byte swizzle
  const uint8_t* dn;          // routed down: bf16 [E][d][I] or codes [E][d][I/2]
  const uint16_t* dn_scales;  // int4 scales [E][d][I/32]
  const uint8_t* sdn;         // shared down bf16 [d][Is]
  const int32_t* sorted_ids;
  const Plan* plan;
  const WorkExpert* work;
  const int32_t* cta;
  const float* h;
  const float* hs;
  float* y;                   // [T*k][d]
  float* ys;                  // [T][d]
  int* status;
  int* dyn;                   // the stage's dynamic-tail ticket counter (DynTail)
  int* dyn_other;             // the gate_up stage's, zeroed here
  int T, d, I, Is, k;
  int rd, rds, xt, stage_bytes, n_stages;
  int stage_off;
  int h_rows;
  SmemPlanArgs sp;
};

// Walks the work experts along a CTA's contiguous unit range.  Units of one
// work expert are numbered group-major (unit = grp * tiles + tile: consecutive
// units share a token group, its activation rows) or, in int4 layers,
// tile-major (unit = tile * groups + grp: an expert with more tokens than a
// unit takes streams each weight tile once from HBM, and its next token groups
// read the tile back from L2 right after).  The work
// experts come from the workspace plan (work != nullptr) or from the CTA's
// shared-memory plan (wex, wnt), where each expert's first unit and first
// sorted position follow from the previous expert's.
struct UnitCursor {
  const WorkExpert* work;  // workspace plan, or nullptr
  const int16_t* wex;      // shared-memory plan: expert ids (-1 = the shared expert)
  const int16_t* wnt;      //   and their token counts
  int n_work, tiles_r, tiles_s, xt;
  bool down;
  bool tile_major;
  int i, ubeg, uend, tiles, groups;
  int expert, n_tok, pos;  // current work expert; pos: its first sorted position
  __device__ __forceinline__ void set(int e, int n) {
    expert = e;
    n_tok = n;
    tiles = e < 0 ? tiles_s : tiles_r;
    groups = (n + xt - 1) / xt;
    uend = ubeg + tiles * groups;
  }
  __device__ __forceinline__ void from_workspace(int idx) {
    const WorkExpert we = work[idx];
    ubeg = down ? we.unit_dn : we.unit_gu;
    pos = we.pos;
    set(we.expert, we.n_tok);
  }
  __device__ __forceinline__ void start(int idx, int ubeg0, int pos0) {
    i = idx;
    if (work) {
      from_workspace(idx);
    } else {
      ubeg = ubeg0;
      pos = pos0;
      set(wex[idx], wnt[idx]);
    }
  }
  __device__ __forceinline__ void advance() {
    ++i;
    if (work) {
      from_workspace(i);
    } else {
      if (expert >= 0) pos += n_tok;
      ubeg = uend;
      set(wex[i], wnt[i]);
    }
  }
  __device__ __forceinline__ void seek(int u) {
    while (u >= uend && i + 1 < n_work) advance();
  }
};

// This CTA's share of a stage: units [u_begin, u_end), starting in work
// expert w0 (first unit ubeg0, first sorted position pos0), of n_work; then
// the stage's dynamic tail [u_dyn, u_total), starting in work expert w_dyn
// (first unit ubeg_dyn, first sorted position pos_dyn).
struct CtaRange {
  int u_begin, u_end, w0, ubeg0, pos0, n_work;
  int u_dyn, u_total, w_dyn, ubeg_dyn, pos_dyn;
};

// The producer's side of a stage's dynamic tail: ticket i of *ctr is unit
// u_dyn + i.  A ticket is fetched ahead of its use (the first two units
// before, the others one), so the atomic's round trip overlaps the copies of
// the units before it.  The counter starts a launch at zero: the other GEMV
// stage of the layer zeroes it, after its dependency wait, in between (gate_up
// zeroes down's, down zeroes gate_up's; every kernel of the layer waits for
// its predecessor to complete before it completes).
struct DynTail {
  int* ctr;
  int u_dyn, u_total;
  int ticket;  // lane 0: the fetched ticket
  __device__ __forceinline__ void fetch(int lane) {
    if (lane == 0) ticket = atomicAdd(ctr, 1);
  }
  __device__ __forceinline__ int take() const {
    return u_dyn + __shfl_sync(0xffffffffu, ticket, 0);
  }
};

// Shared-memory word of each stage holding the unit the producer put there,
// for the units of the dynamic tail (-1: no more units).
constexpr int kStageUnitOff = 192;  // inside the barrier area, after the barriers

// The producer's last stage (its j-th): no unit, so that the consumers, which
// learn the tail's units from the stages, stop.  Clears ok if the wait for the
// slot gives up.
__device__ __forceinline__ void end_of_units(uint64_t* full, uint64_t* empty, int* s_unit, int j,
                                             int NS, int lane, int* status, bool& ok) {
  const int s = j % NS, use = j / NS;
  if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), status)) {
    ok = false;
    return;
  }
  if (lane == 0) {
    s_unit[s] = -1;
    mbar_arrive(&full[s]);
  }
  __syncwarp();
}

// Ints of shared-memory scratch smem_plan needs (it lives in the stage ring,
// before the first copy is issued).
__host__ __device__ constexpr int smem_plan_scratch_ints(int S, int E, int T) {
  return S + E * ((T + 31) / 32) + 2 * E + 3 * (E + 2) + 32 * 5;
}

// floor(n / d) for 0 <= n < 2^22 and d >= 1, given inv = 1.0f / d: (n + 1/2)
// / d lies at least 1/(2d) from an integer, and the two float roundings move
// it by less than (n / d) 2^-23 < 1/(2d).
__device__ __forceinline__ int div_small(int n, float inv) {
  return (int)(((float)n + 0.5f) * inv);
}

// The most experts one thread of a plan-building CTA owns (E <= 1024 over the
// 160 threads of the expert kernels).
constexpr int kPlanRun = 8;

// smem_plan for S = T k <= 64 slots, on one warp (lane = threadIdx.x < 32):
// the same work list, sorted positions and aligned-layout slice.  Keys
// (expert << 12 | slot) of the 64 positions i = lane + 32 r sit two per lane
// and go through a bitonic sort network (in-lane at distance 32, shuffles
// below); invalid ids sort last and count nowhere.  A run of one expert starts
// where the expert changes; its work index is the number of run starts below
// it, its first sorted position is its index in the sorted keys.  Results in
// shared memory: wex, wnt, u0, c0, p0 per work expert, poe (padded offset) per
// routed work expert, sorted; n_work / units / cost returned in every lane.
__device__ __forceinline__ void warp_plan(const SmemPlanArgs& sp, int S, int E, int B, int T,
                                          int xt, int tiles_r, int tiles_s, int base, int base_s,
                                          int tw, bool shared_expert, int eb, int ee,
                                          int16_t* wex, int16_t* wnt, int32_t* sorted, int* poe,
                                          int* u0, int* c0, int* p0, int& n_work, int& units,
                                          int& cost, int* status) {
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kNone = 0x7fffffff;
  const int lane = threadIdx.x & 31;
  const float inv_xt = 1.0f / (float)xt, inv_b = 1.0f / (float)B;
  int key[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int slot = lane + 32 * r;
    int v = kNone;
    if (slot < S) {
      const int e = __ldcg(sp.ids + slot);
      if (e < 0 || e >= E)
        record_status(status, kStatusDeviceCheck);
      else
        v = (e << 12) | slot;
    }
    key[r] = v;
  }
  // Bitonic network over i = lane + 32 r: blocks of `size` alternate
  // ascending / descending until the last (size 64) sorts all ascending.
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 32) {
        const int lo = min(key[0], key[1]), hi = max(key[0], key[1]);
        key[0] = lo;
        key[1] = hi;
      } else {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int i = lane + 32 * r;
          const int other = __shfl_xor_sync(kAll, key[r], stride);
          const bool up = (i & size) == 0, lower = (i & stride) == 0;
          key[r] = lower == up ? min(key[r], other) : max(key[r], other);
        }
      }
    }
  }
  int ex[2], sl[2];
  bool val[2], head[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    val[r] = key[r] != kNone;
    ex[r] = key[r] >> 12;
    sl[r] = key[r] & 4095;
  }
  int prev0 = __shfl_up_sync(kAll, ex[0], 1), prev1 = __shfl_up_sync(kAll, ex[1], 1);
  const int last0 = __shfl_sync(kAll, ex[0], 31);
  if (lane == 0) {
    prev0 = -1;
    prev1 = last0;
  }
  head[0] = val[0] && ex[0] != prev0;
  head[1] = val[1] && ex[1] != prev1;
  const uint64_t H = (uint64_t)__ballot_sync(kAll, head[1]) << 32 | __ballot_sync(kAll, head[0]);
  const int nvalid = __popc(__ballot_sync(kAll, val[0])) + __popc(__ballot_sync(kAll, val[1]));
  const int nw = __popcll(H);
  // Per run start: rows after padding, units, cost; exclusive scans in i order.
  int q[2][3];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = lane + 32 * r;
    q[r][0] = q[r][1] = q[r][2] = 0;
    if (head[r]) {
      const uint64_t above = i == 63 ? 0ull : H >> (i + 1);
      const int c = above ? __ffsll((long long)above) : nvalid - i;
      const int g = div_small(c + xt - 1, inv_xt);
      q[r][0] = div_small(c + B - 1, inv_b) * B;
      q[r][1] = tiles_r * g;
      q[r][2] = tiles_r * (g * base + tw * c);
    }
  }
  int xs[2][3], tot[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    int inc0 = q[0][j], inc1 = q[1][j];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n0 = __shfl_up_sync(kAll, inc0, o), n1 = __shfl_up_sync(kAll, inc1, o);
      if (lane >= o) {
        inc0 += n0;
        inc1 += n1;
      }
    }
    const int t0 = __shfl_sync(kAll, inc0, 31);
    xs[0][j] = inc0 - q[0][j];
    xs[1][j] = t0 + inc1 - q[1][j];
    tot[j] = t0 + __shfl_sync(kAll, inc1, 31);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = lane + 32 * r;
    if (val[r]) sorted[i] = sl[r];
    if (head[r]) {
      const uint64_t above = i == 63 ? 0ull : H >> (i + 1);
      const int c = above ? __ffsll((long long)above) : nvalid - i;
      const int idx = __popcll(H & ((1ull << i) - 1ull));
      wex[idx] = (int16_t)ex[r];
      wnt[idx] = (int16_t)c;
      u0[idx] = xs[r][1];
      c0[idx] = xs[r][2];
      p0[idx] = i;
      poe[idx] = xs[r][0];
    }
  }
  n_work = nw;
  units = tot[1];
  cost = tot[2];
  if (shared_expert) {
    const int sg = div_small(T + xt - 1, inv_xt);
    if (lane == 0) {
      wex[nw] = -1;
      wnt[nw] = (int16_t)T;
      u0[nw] = units;
      c0[nw] = cost;
      p0[nw] = 0;
    }
    n_work += 1;
    units += tiles_s * sg;
    cost += tiles_s * (sg * base_s + T);
  }
  __syncwarp();
  int32_t* const abi_sorted = sp.sorted_ids;
  if (abi_sorted == nullptr) return;
  // This CTA's slice [eb, ee) of the aligned layout.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = lane + 32 * r;
    if (val[r] && ex[r] >= eb && ex[r] < ee) {
      const uint64_t at_or_below = i == 63 ? ~0ull : (2ull << i) - 1ull;
      const int idx = __popcll(H & at_or_below) - 1;
      abi_sorted[poe[idx] + (i - p0[idx])] = sl[r];
    }
  }
  for (int e = eb + lane; e < ee; e += 32) {
    // Padded offset of expert e: that of the first touched expert >= e.
    int lo = 0, hi = nw;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (wex[mid] < e) lo = mid + 1; else hi = mid;
    }
    const int off = lo < nw ? poe[lo] : tot[0];
    sp.expert_offsets[e] = off;
    if (lo < nw && wex[lo] == e) {
      const int c = wnt[lo];
      const int P = div_small(c + B - 1, inv_b) * B;
      for (int rr = c; rr < P; ++rr) abi_sorted[off + rr] = S;  // padding
      for (int b = 0; b < P; b += B) sp.block_ids[div_small(off + b, inv_b)] = e;
    }
  }
  if (blockIdx.x == 0 && lane == 0) {
    sp.expert_offsets[E] = tot[0];
    *sp.num_post_pad = tot[0];
  }
}

// The plan of one expert stage, built in shared memory by all threads of the
// CTA from the routing ids (decode sizes: T <= 128, E <= 1024): the align
// step's counting sort by expert in arrival order, the work list (touched
// experts in ascending id, then the shared expert) and this CTA's unit range
// -- the split the workspace plan gives: CTA c starts where the running
// estimated cost reaches c / grid of the stage's total.  Every CTA derives the
// same plan from the same ids.
// A token's k experts are distinct, so a slot's rank within its expert (its
// arrival order) is the number of earlier TOKENS that chose the expert: each
// expert keeps a bitmask over the tokens, set with one shared-memory atomicOr
// per slot, and a rank is the popcount of the bits below the token.  Each
// thread owns a run of at most kPlanRun experts; one block scan gives the
// work indices, first units, costs and positions.  The steps are
// latency-bound, so the code keeps the dependent chain short: counts cached
// in registers, float-reciprocal divisions, four barriers.
// Persistent results: wex, wnt ([n_work]) and sorted ([T*k]: each expert's
// slots at its running position, no padding).  With sp.sorted_ids, the CTA
// also writes its slice of the aligned layout (moe_align_block_size) to the
// workspace: the experts [blockIdx.x * E / grid, (blockIdx.x + 1) * E / grid).
// The CTA's range is left in `range` (shared memory).
__device__ void smem_plan(CtaRange& range, const SmemPlanArgs sp, int T, int k, bool shared_expert,
                              int tiles_r, int tiles_s, int xt, int16_t* wex, int16_t* wnt,
                              int32_t* sorted, int* scratch, int* status) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int S = T * k, E = sp.E, B = sp.B, W = (T + 31) >> 5;
  const int base = sp.base, base_s = sp.base_s, tw = sp.tok_w;
  int32_t* const abi_sorted = sp.sorted_ids;
  const float inv_k = 1.0f / (float)k, inv_xt = 1.0f / (float)xt, inv_b = 1.0f / (float)B;
  // This CTA's slice of the aligned layout (E * grid < 2^31).
  const int eb = (int)(blockIdx.x * (unsigned)E / gridDim.x);
  const int ee = (int)((blockIdx.x + 1) * (unsigned)E / gridDim.x);
  int* s_ids = scratch;                                     // [S]
  uint32_t* mask = reinterpret_cast<uint32_t*>(s_ids + S);  // [E][W] tokens of each expert
  int* p0e = reinterpret_cast<int*>(mask + E * W);          // [E] first sorted position
  int* poe = p0e + E;                                       // [E] padded offset
  int* u0 = poe + E;                                        // [E + 2] first unit of a work expert
  int* c0 = u0 + E + 2;                                     // [E + 2] cost before a work expert
  int* p0 = c0 + E + 2;                                     // [E + 2] its first sorted position
  int* scan = p0 + E + 2;                                   // [32 * 5]
  int n_work = 0, units = 0, cost = 0;  // warp 0 (tid < 3) reads them below
  if (S <= 64) {
    // Up to 64 slots: one warp sorts the (expert, slot) keys -- slot order
    // within an expert is arrival order -- finds the runs by ballot and sums
    // their rows, units and costs with warp scans; no block barrier.
    if (tid < 32) warp_plan(sp, S, E, B, T, xt, tiles_r, tiles_s, base, base_s, tw, shared_expert,
                            eb, ee, wex, wnt, sorted, poe, u0, c0, p0, n_work, units, cost,
                            status);
  } else {
    for (int s = tid; s < S; s += nthr) {
      int e = __ldcg(sp.ids + s);
      if (e < 0 || e >= E) {
        record_status(status, kStatusDeviceCheck);
        e = -1;
      }
      s_ids[s] = e;
    }
    for (int i = tid; i < E * W; i += nthr) mask[i] = 0u;
    __syncthreads();
    for (int s = tid; s < S; s += nthr) {
      const int e = s_ids[s];
      const int t = div_small(s, inv_k);
      if (e >= 0) atomicOr(&mask[e * W + (t >> 5)], 1u << (t & 31));
    }
    __syncthreads();
    // Thread-owned experts [e0, e0 + n): counts, then per expert padded rows,
    // touched, units, cost, tokens.
    const int run = (E + nthr - 1) / nthr;
    const int e0 = min(E, tid * run), n = min(E, e0 + run) - e0;
    int cnt[kPlanRun];
    int loc[5] = {0, 0, 0, 0, 0};
  #pragma unroll
    for (int i = 0; i < kPlanRun; ++i) {
      int c = 0;
      if (i < n)
        for (int w = 0; w < W; ++w) c += __popc(mask[(e0 + i) * W + w]);
      cnt[i] = c;
      const int g = div_small(c + xt - 1, inv_xt);
      loc[0] += div_small(c + B - 1, inv_b) * B;
      loc[1] += c > 0 ? 1 : 0;
      loc[2] += tiles_r * g;
      loc[3] += tiles_r * (g * base + tw * c);
      loc[4] += c;
    }
    int ex[5], tot[5];
    block_scan<5>(loc, ex, tot, scan);
  #pragma unroll
    for (int i = 0; i < kPlanRun; ++i) {
      const int c = cnt[i], e = e0 + i;
      const int g = div_small(c + xt - 1, inv_xt);
      const int P = div_small(c + B - 1, inv_b) * B;
      if (c > 0) {
        const int idx = ex[1];
        wex[idx] = (int16_t)e;
        wnt[idx] = (int16_t)c;
        u0[idx] = ex[2];
        c0[idx] = ex[3];
        p0[idx] = ex[4];
        p0e[e] = ex[4];
        poe[e] = ex[0];
        if (abi_sorted != nullptr && e >= eb && e < ee) {
          for (int r = c; r < P; ++r) abi_sorted[ex[0] + r] = S;  // padding
          for (int b = 0; b < P; b += B) sp.block_ids[div_small(ex[0] + b, inv_b)] = e;
        }
      }
      if (abi_sorted != nullptr && i < n && e >= eb && e < ee) sp.expert_offsets[e] = ex[0];
      ex[0] += P;
      ex[1] += c > 0 ? 1 : 0;
      ex[2] += tiles_r * g;
      ex[3] += tiles_r * (g * base + tw * c);
      ex[4] += c;
    }
    n_work = tot[1];
    units = tot[2];
    cost = tot[3];
    if (shared_expert) {
      const int sg = div_small(T + xt - 1, inv_xt);
      if (tid == 0) {
        wex[n_work] = -1;
        wnt[n_work] = (int16_t)T;
        u0[n_work] = units;
        c0[n_work] = cost;
        p0[n_work] = 0;
      }
      n_work += 1;
      units += tiles_s * sg;
      cost += tiles_s * (sg * base_s + T);
    }
    if (abi_sorted != nullptr && blockIdx.x == 0 && tid == 0) {
      sp.expert_offsets[E] = tot[0];
      *sp.num_post_pad = tot[0];
    }
    __syncthreads();
    // Each slot at its expert's running position (arrival order: the earlier
    // tokens of the expert come first); this CTA's slice of the aligned layout.
    for (int s = tid; s < S; s += nthr) {
      const int e = s_ids[s];
      if (e < 0) continue;
      const int t = div_small(s, inv_k);
      const uint32_t* m = mask + e * W;
      int r = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
      for (int w = 0; w < (t >> 5); ++w) r += __popc(m[w]);
      sorted[p0e[e] + r] = s;
      if (abi_sorted != nullptr && e >= eb && e < ee) abi_sorted[poe[e] + r] = s;
    }
  }
  // This CTA's range: the start of CTA c and of CTA c + 1, and the start of
  // the dynamic tail (CTA grid).
  if (tid < 3) {
    const int c = tid < 2 ? (int)blockIdx.x + tid : (int)gridDim.x;
    int u = 0, w = 0;
    if (c == (int)gridDim.x && !sp.tail) {
      u = units;
      w = n_work > 0 ? n_work - 1 : 0;
    } else if (c > 0 && n_work > 0) {
      const int target =
          split_target(c, gridDim.x, cost, sp.tail != 0,
                       sp.sorted_ids != nullptr && !sp.tail ? kDownSkew : 0.f);
      int lo = 0, hi = n_work - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (c0[mid] <= target) lo = mid; else hi = mid - 1;
      }
      w = lo;
      const bool sh = shared_expert && lo == n_work - 1;
      u = unit_at_cost(target, c0[lo], u0[lo], sh ? tiles_s : tiles_r, wnt[lo], xt,
                       sh ? base_s : base, sh ? 1 : tw, sp.tile_major != 0);
    }
    if (tid == 0) {
      range.u_begin = u;
      range.w0 = w;
      range.ubeg0 = u0[w];
      range.pos0 = p0[w];
      range.n_work = n_work;
    } else if (tid == 1) {
      range.u_end = u;
    } else {
      range.u_dyn = u;
      range.u_total = units;
      range.w_dyn = w;
      range.ubeg_dyn = u0[w];
      range.pos_dyn = p0[w];
    }
  }
  __syncthreads();
}

// Tiled 2D tensor copy of the box at (x, y) into shared memory, completion as
// transaction bytes on `bar`, with an L2 cache policy.
__device__ __forceinline__ void tma_box_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                           uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Tiled 3D tensor copy of the box at (x, y, z).
__device__ __forceinline__ void tma_box_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                           int z, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------ smem loads
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_bf16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __uint_as_float((uint32_t)v << 16);
}

// ------------------------------------------------------------------ dot pieces
// Packed fp32 pairs (element 2j in the low word, 2j + 1 in the high word): one
// instruction does both lanes' fma / sub, each rounded as the scalar would be.
__device__ __forceinline__ uint64_t f2(uint32_t lo, uint32_t hi) {
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ float f2sum(uint64_t v) {
  return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}

// Two bf16 (element 2j low, 2j + 1 high) as an fp32 pair.
__device__ __forceinline__ uint64_t bf16x2_f2(uint32_t w) { return f2(w << 16, w & 0xffff0000u); }

// ------------------------------------------------------------------ int4 on the tensor pipe
// Token rows of an int4 layer sit at a pitch 16 bytes beyond the row: that
// shifts consecutive rows by four banks, so the eight rows one load reads fall
// on distinct banks.
__host__ __device__ constexpr int x_pitch(int fmt, int d) { return fmt ? 2 * d + 16 : 2 * d; }
// Bytes of the cross-warp partial sums of the int4 gate_up consumers: two
// buffers x three warps x 32 lanes x 4 floats.
constexpr int kI4RedBytes = 2 * 3 * 32 * 16;

// Four exact bf16 pairs from one word of eight int4 codes (element j in nibble
// j, stored as code + 8): pair i = (code i, code i + 4), low half first.  The
// two nibbles land in the mantissa of 128.0 (bf16 0x4300, mantissa step 1) by
// one shift and one and-or; one packed fma then takes 136 = 128 + 8 off both
// halves, exactly.
__device__ __forceinline__ void dequant_pairs(uint32_t v, uint32_t (&q)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t biased = ((v >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;"
        : "=r"(q[i])
        : "r"(biased), "r"(0x3F803F80u), "r"(0xC308C308u));  // x * 1 - 136
  }
}

// D = A B + C on the tensor pipe: 16x16 bf16 A (row-major fragment), 16x8 bf16
// B (column fragment), fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// int4 gate_up stage of RG rows (8 or 16): the unit's RG gate code rows arrive
// as one tensor box of d / 256 chunks x RG rows x 128 bytes (chunk-major) with
// the 128-byte swizzle, the RG up rows as a second, then their scales densely
// (gate, up), then the tokens' x rows.  Chunk c of a row holds groups 8c ..
// 8c + 7 of 32 codes, 16 bytes each; group 8c + i of row r sits in slot
// i ^ (r % 8) of the row's 128 bytes.
__host__ __device__ constexpr int i4g_box_bytes(int d, int rg) { return rg * d / 2; }
__host__ __device__ constexpr int i4g_weight_bytes(int d, int rg) { return rg * (d + d / 8); }

// One consumer warp's share of an int4 gate_up unit on the tensor pipe: rows
// r8 .. r8 + 7 of the unit's gate and up rows, over the 8-group chunks c = c0,
// c0 + cstep, ... of d.  The share is one 16x8 product per 16 codes: A = the
// gate rows on tile rows 0..7, the up rows on 8..15; B = the tokens'
// activations; lane (g, t) = (lane / 4, lane % 4) holds, in acc, gate and up
// row r8 + g for tokens 2t and 2t + 1 -- both halves of a SwiGLU.
// Within a group of 32, thread t takes its code word t (codes 8t .. 8t + 7) and
// the tile's k positions map onto them as (8t, 8t + 4), (8t + 1, 8t + 5) for the
// first product and (8t + 2, 8t + 6), (8t + 3, 8t + 7) for the second; the
// activations are permuted to match.  Each group's two products start from
// zero and are scaled by the rows' bf16 scales into the fp32 accumulators: per
// group, the sum of code x activation, then x scale (the definition regrouped,
// exact up to rounding order).
// codes: the stage (RG rows per box); sg, su: the gate and up scales of row
// r8 + g; xr: token g's row at thread t's 16 bytes.
__device__ __forceinline__ void gu_int4_mma(uint32_t codes, int d, int RG, int r8, int g, int t,
                                            uint32_t sg, uint32_t su, uint32_t xr, bool has_x,
                                            int c0, int cstep, float (&acc)[4]) {
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  const int nc = d / 256;
  const uint32_t up = (uint32_t)i4g_box_bytes(d, RG);
  for (int c = c0; c < nc; c += cstep) {
    const uint4 sgv = lds128(sg + 16u * c), suv = lds128(su + 16u * c);
    const uint32_t crow = codes + (uint32_t)((c * RG + r8 + g) * 128 + 4 * t);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t ca = crow + (uint32_t)((i ^ g) << 4);
      uint32_t vg, vu;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(vg) : "r"(ca));
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(vu) : "r"(ca + up));
      const uint32_t wg = (i < 2 ? sgv.x : i < 4 ? sgv.y : i < 6 ? sgv.z : sgv.w);
      const uint32_t wu = (i < 2 ? suv.x : i < 4 ? suv.y : i < 6 ? suv.z : suv.w);
      const float fg = __uint_as_float(i & 1 ? wg & 0xffff0000u : wg << 16);
      const float fu = __uint_as_float(i & 1 ? wu & 0xffff0000u : wu << 16);
      const uint4 xv = has_x ? lds128(xr + 64u * (8 * c + i)) : make_uint4(0u, 0u, 0u, 0u);
      uint32_t qg[4], qu[4];
      dequant_pairs(vg, qg);
      dequant_pairs(vu, qu);
      const uint32_t b10 = __byte_perm(xv.x, xv.z, 0x5410), b11 = __byte_perm(xv.x, xv.z, 0x7632);
      const uint32_t b20 = __byte_perm(xv.y, xv.w, 0x5410), b21 = __byte_perm(xv.y, xv.w, 0x7632);
      float p[4];
      mma_16816(p, qg[0], qu[0], qg[1], qu[1], b10, b11, zero);
      mma_16816(p, qg[2], qu[2], qg[3], qu[3], b20, b21, p);
      acc[0] = fmaf(p[0], fg, acc[0]);
      acc[1] = fmaf(p[1], fg, acc[1]);
      acc[2] = fmaf(p[2], fu, acc[2]);
      acc[3] = fmaf(p[3], fu, acc[3]);
    }
  }
}

// int4 down stage: the unit's 128 code rows of W_down arrive as I / 256 tensor
// boxes of 128 rows x 128 bytes with the 128-byte swizzle (16-byte chunk c of
// row r stored at chunk c ^ (r % 8): the eight rows one load reads fall on
// distinct banks), then the rows' scales densely, then the tokens' h rows.
constexpr int kI4DnRows = 128;
constexpr int kI4DnBox = kI4DnRows * 128;  // bytes of one code box
__host__ __device__ constexpr int i4d_codes_bytes(int I) { return (I / 256) * kI4DnBox; }
__host__ __device__ constexpr int i4d_h_pitch(int I) { return 2 * I + 16; }

// Shared address of code word t of group gi of row r in a swizzled box set.
__device__ __forceinline__ uint32_t i4d_code_addr(uint32_t codes, int r, int gi, int t) {
  return codes + (uint32_t)((gi >> 3) * kI4DnBox + r * 128 + (((gi & 7) ^ (r & 7)) << 4) + 4 * t);
}

// Column of element c of an int4 layer's h row: each 8-element block is
// stored in the order 0, 4, 1, 5, 2, 6, 3, 7 -- the k pairs (i, i + 4) of the
// nibble pairing -- so that one 16-byte load is the four B registers of a
// group's two down products, with no permute.
__device__ __forceinline__ int i4h_col(int c) { return (c & ~7) | ((c & 3) << 1) | ((c >> 2) & 1); }

// One consumer warp's m16 tile of an int4 down unit: rows ra and rb (the
// tile's rows g and g + 8 of lane (g, t)), all I / 32 groups, up to 8 tokens.
// In an int4 layer h travels as two bf16 planes, hi = bf16(h) and lo = bf16(h
// - hi), and each group takes one product on each (the pair carries h to about
// 2^-17): the k positions map onto the codes as in gu_int4_mma, and the h
// rows are stored in that order (i4h_col).  acc: rows ra, rb x tokens 2t,
// 2t + 1.
__device__ __forceinline__ void dn_int4_mma(uint32_t codes, int ra, int rb, int t, uint32_t sa,
                                            uint32_t sb, uint32_t hh, uint32_t hl, bool has_h,
                                            int ng, float (&acc)[4]) {
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int gi = 0; gi < ng; ++gi) {
    uint32_t va, vb;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(va) : "r"(i4d_code_addr(codes, ra, gi, t)));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(vb) : "r"(i4d_code_addr(codes, rb, gi, t)));
    const float fa = lds_bf16(sa + 2u * gi), fb = lds_bf16(sb + 2u * gi);
    const uint4 H = has_h ? lds128(hh + 64u * gi) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 L = has_h ? lds128(hl + 64u * gi) : make_uint4(0u, 0u, 0u, 0u);
    uint32_t qa[4], qb[4];
    dequant_pairs(va, qa);
    dequant_pairs(vb, qb);
    float p[4];
    mma_16816(p, qa[0], qb[0], qa[1], qb[1], H.x, H.y, zero);
    mma_16816(p, qa[2], qb[2], qa[3], qb[3], H.z, H.w, p);
    mma_16816(p, qa[0], qb[0], qa[1], qb[1], L.x, L.y, p);
    mma_16816(p, qa[2], qb[2], qa[3], qb[3], L.z, L.w, p);
    acc[0] = fmaf(p[0], fa, acc[0]);
    acc[1] = fmaf(p[1], fa, acc[1]);
    acc[2] = fmaf(p[2], fb, acc[2]);
    acc[3] = fmaf(p[3], fb, acc[3]);
  }
}

// bf16 of v, round to nearest even, as raw bits.
__device__ __forceinline__ uint16_t bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// ------------------------------------------------------------------ gate_up math
// One warp: gate row at wg, up row at wu (shared addresses), NT token rows at
// xa + q * xs.  bf16 weights; 16-byte chunks strided over the lanes.  Returns
// the per-token full dot products in every lane.
// The (even, odd) products of each bf16 pair go into an fp32 pair with one
// packed fma: the order of the sums is that of two scalar accumulators.
template <int NT>
__device__ __forceinline__ void gu_rows_bf16(uint32_t wg, uint32_t wu, uint32_t xa, uint32_t xs,
                                             int nch, int lane, float* g, float* u) {
  uint64_t pg[NT], pu[NT];
#pragma unroll
  for (int q = 0; q < NT; ++q) pg[q] = pu[q] = 0ull;
#pragma unroll 2
  for (int c = lane; c < nch; c += 32) {
    const uint32_t off = (uint32_t)c * 16u;
    const uint4 vg = lds128(wg + off), vu = lds128(wu + off);
    const uint64_t g0 = bf16x2_f2(vg.x), g1 = bf16x2_f2(vg.y), g2 = bf16x2_f2(vg.z),
                   g3 = bf16x2_f2(vg.w);
    const uint64_t u0 = bf16x2_f2(vu.x), u1 = bf16x2_f2(vu.y), u2 = bf16x2_f2(vu.z),
                   u3 = bf16x2_f2(vu.w);
    uint4 xv[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) xv[q] = lds128(xa + q * xs + off);
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const uint64_t x0 = bf16x2_f2(xv[q].x), x1 = bf16x2_f2(xv[q].y), x2 = bf16x2_f2(xv[q].z),
                     x3 = bf16x2_f2(xv[q].w);
      pg[q] = ffma2(g0, x0, pg[q]);
      pu[q] = ffma2(u0, x0, pu[q]);
      pg[q] = ffma2(g1, x1, pg[q]);
      pu[q] = ffma2(u1, x1, pu[q]);
      pg[q] = ffma2(g2, x2, pg[q]);
      pu[q] = ffma2(u2, x2, pu[q]);
      pg[q] = ffma2(g3, x3, pg[q]);
      pu[q] = ffma2(u3, x3, pu[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    g[q] = warp_sum(f2sum(pg[q]));
    u[q] = warp_sum(f2sum(pu[q]));
  }
}

// One consumer warp's share of a bf16 gate_up unit: NT tokens; lane q writes
// token q's h value at hout + q * hstride.
template <int NT>
__device__ __forceinline__ void gu_warp(uint32_t wg, uint32_t wu, uint32_t xa, uint32_t xs, int d,
                                        int lane, float* hout, size_t hstride) {
  float g[NT], u[NT];
  gu_rows_bf16<NT>(wg, wu, xa, xs, d / 8, lane, g, u);
  float gv = g[0], uv = u[0];
#pragma unroll
  for (int q = 1; q < NT; ++q)
    if (lane == q) {
      gv = g[q];
      uv = u[q];
    }
  if (lane < NT) hout[(size_t)lane * hstride] = silu(gv) * uv;
}

// ------------------------------------------------------------------ down math
// Two bf16 weight rows (wa, wb) per 8-lane group, so every h chunk loaded from
// shared memory serves both.  NT tokens' h rows (fp32) at ha + q * hsb.  On
// return, lane sl of the group holds token sl's outputs for both rows.
template <int NT>
__device__ __forceinline__ void dn_rows2(uint32_t wa, uint32_t wb, uint32_t ha, uint32_t hsb,
                                         int Iw, int sl, float& oa, float& ob) {
  float a0[NT], a1[NT], b0[NT], b1[NT];
  // (even, odd) pairs with packed fmas: the sums of a0/a1 and b0/b1 in order.
  uint64_t pa[NT], pb[NT];
#pragma unroll
  for (int q = 0; q < NT; ++q) pa[q] = pb[q] = 0ull;
#pragma unroll 2
  for (int c = sl; c < Iw / 8; c += 8) {
    const uint32_t off = (uint32_t)c * 16u;
    const uint4 va = lds128(wa + off), vb = lds128(wb + off);
    const uint64_t wa0 = bf16x2_f2(va.x), wa1 = bf16x2_f2(va.y), wa2 = bf16x2_f2(va.z),
                   wa3 = bf16x2_f2(va.w);
    const uint64_t wb0 = bf16x2_f2(vb.x), wb1 = bf16x2_f2(vb.y), wb2 = bf16x2_f2(vb.z),
                   wb3 = bf16x2_f2(vb.w);
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      // Lanes sl >= 4 load the chunk's upper 16 bytes first (the lanes' h
      // chunks are 32 bytes apart: this puts one load's lanes on distinct
      // banks); the products are taken in the same order either way.
      const uint32_t hb = ha + q * hsb + 2u * off;
      const bool up = (sl >> 2) & 1;
      const float4 first = lds128f(hb + (up ? 16u : 0u));
      const float4 second = lds128f(hb + (up ? 0u : 16u));
      const float4 hp = up ? second : first, hq = up ? first : second;
      const uint64_t h0 = f2(__float_as_uint(hp.x), __float_as_uint(hp.y));
      const uint64_t h1 = f2(__float_as_uint(hp.z), __float_as_uint(hp.w));
      const uint64_t h2 = f2(__float_as_uint(hq.x), __float_as_uint(hq.y));
      const uint64_t h3 = f2(__float_as_uint(hq.z), __float_as_uint(hq.w));
      pa[q] = ffma2(wa0, h0, pa[q]);
      pb[q] = ffma2(wb0, h0, pb[q]);
      pa[q] = ffma2(wa1, h1, pa[q]);
      pb[q] = ffma2(wb1, h1, pb[q]);
      pa[q] = ffma2(wa2, h2, pa[q]);
      pb[q] = ffma2(wb2, h2, pb[q]);
      pa[q] = ffma2(wa3, h3, pa[q]);
      pb[q] = ffma2(wb3, h3, pb[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    a0[q] = __uint_as_float((uint32_t)pa[q]);
    a1[q] = __uint_as_float((uint32_t)(pa[q] >> 32));
    b0[q] = __uint_as_float((uint32_t)pb[q]);
    b1[q] = __uint_as_float((uint32_t)(pb[q] >> 32));
  }
  oa = ob = 0.f;
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    float va = a0[q] + a1[q], vb = b0[q] + b1[q];
    va += __shfl_xor_sync(0xffffffffu, va, 4);
    vb += __shfl_xor_sync(0xffffffffu, vb, 4);
    va += __shfl_xor_sync(0xffffffffu, va, 2);
    vb += __shfl_xor_sync(0xffffffffu, vb, 2);
    va += __shfl_xor_sync(0xffffffffu, va, 1);
    vb += __shfl_xor_sync(0xffffffffu, vb, 1);
    if (sl == q) {
      oa = va;
      ob = vb;
    }
  }
}

// Producer drain after an abort: wait (bounded) for the last fills of every
// stage so no bulk copy is still writing shared memory when the CTA exits.
__device__ void drain_stages(uint64_t* full, int issued, int n_stages, int* status) {
  for (int j = max(0, issued - n_stages); j < issued; ++j)
    mbar_wait(&full[j % n_stages], (uint32_t)((j / n_stages) & 1), status);
}

// --------------------------------------------------------------------------- gate_up
// This CTA's 16-byte-aligned slice of [p, p + bytes) (bytes a multiple of 16),
// prefetched into L2 in pieces of at most 64 KB.
__device__ __forceinline__ void prefetch_slice_l2(const uint8_t* p, size_t bytes) {
  if (p == nullptr) return;
  const size_t per = (ceil_div(bytes, (size_t)gridDim.x) + 15) & ~(size_t)15;
  const size_t b0 = per * blockIdx.x;
  const size_t b1 = min(bytes, b0 + per);
  for (size_t b = b0; b < b1; b += 65536)
    bulk_prefetch_l2(p + b, (uint32_t)min((size_t)65536, b1 - b));
}

// Shared-memory layout of both expert kernels: barriers (kBarBytes), then
// (shared-memory plan only) the persistent plan -- wex int16 [E + 1], wnt
// int16 [E + 1], sorted int32 [T*k] -- then, at stage_off, the stage ring, whose
// start also holds smem_plan's scratch until the first copy is issued.
__device__ __forceinline__ void plan_arrays(uint8_t* smem, int E, int16_t*& wex, int16_t*& wnt,
                                            int32_t*& sorted) {
  const int wb = (int)round_up(2 * (E + 1), 16);
  wex = reinterpret_cast<int16_t*>(smem + kBarBytes);
  wnt = reinterpret_cast<int16_t*>(smem + kBarBytes + wb);
  sorted = reinterpret_cast<int32_t*>(smem + kBarBytes + 2 * wb);
}

template <int kFmt, bool kTail>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    gate_up_kernel(const __grid_constant__ GuArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* red_full = empty + kMaxStages;  // [2] int4 partial-sum hand-off
  uint64_t* red_empty = red_full + 2;       // [2]
  // int4: the ring starts on a 1024-byte boundary (the swizzled code boxes).
  const uint32_t ring_pad =
      kFmt ? ((1024u - ((smem_u32(smem) + (uint32_t)a.stage_off) & 1023u)) & 1023u) : 0u;
  uint8_t* stages = smem + a.stage_off + ring_pad;
  const uint32_t stages_sa = smem_u32(stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.n_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      // int4: warps tp + ntile j (j >= 1) hand their partial sums to warp tp.
      const int ntile = a.rg / 8;
      mbar_init(&red_full[b], kConsumerWarps - ntile);
      mbar_init(&red_empty[b], ntile);
    }
    fence_barrier_init();
  }
  // The shared expert's weights do not depend on the routing: each CTA
  // prefetches its slice of them into L2 while the routing kernel still runs
  // and HBM is otherwise idle, which takes their reads out of the weight stream
  // of this stage and the next.
  if (threadIdx.x == kConsumerWarps * 32 && a.sgu != nullptr) {
    prefetch_slice_l2(a.sgu, (size_t)4 * a.Is * a.d);
    prefetch_slice_l2(a.sdn, (size_t)2 * a.Is * a.d);
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.dyn_other = 0;

  // The stall test hook (moe_workspace_inject_stall): the producer issues
  // nothing and the consumers' waits give up after the armed limit.
  const int stall_us = a.status ? __ldcg(a.status + kStallWord) : 0;
  const uint64_t wait_ns = stall_us > 0 ? (uint64_t)stall_us * 1000u : kWaitLimitNs;

  const int d = a.d;
  const int xt = a.xt;
  // Routed row bytes (codes only, for int4) and int4 scale bytes per row; the
  // token rows' pitch in a stage.
  const int rowb = kFmt ? d / 2 : d * 2;
  const int srowb = kFmt ? d / 16 : 0;
  const int xp = x_pitch(kFmt, d);
  UnitCursor cur;
  cur.tiles_r = (int)ceil_div(a.I, a.rg);
  cur.tiles_s = a.Is > 0 ? (int)ceil_div(a.Is, a.rgs) : 1;
  cur.xt = xt;
  cur.down = false;
  cur.tile_major = kFmt != 0;
  // This CTA's range, in shared memory (read where needed, not held in
  // registers across the unit loops).
  __shared__ CtaRange rg;
  const int32_t* sorted;  // sorted position -> slot (shared or global memory)
  if (a.sp.ids != nullptr) {
    int16_t *wex, *wnt;
    int32_t* ss;
    plan_arrays(smem, a.sp.E, wex, wnt, ss);
    cur.work = nullptr;
    cur.wex = wex;
    cur.wnt = wnt;
    smem_plan(rg, a.sp, a.T, a.k, a.Is > 0, cur.tiles_r, cur.tiles_s, xt, wex, wnt, ss,
                   reinterpret_cast<int*>(stages), a.status);
    sorted = ss;
  } else {
    cur.work = a.work;
    if (threadIdx.x == 0) {
      rg.n_work = a.plan->n_work;
      rg.u_begin = a.cta[blockIdx.x];
      rg.u_end = a.cta[blockIdx.x + 1];
      rg.w0 = a.cta[gridDim.x + 1 + blockIdx.x];
      rg.ubeg0 = rg.pos0 = 0;
      rg.u_dyn = a.cta[gridDim.x];
      rg.w_dyn = a.cta[2 * gridDim.x + 1];
      rg.ubeg_dyn = rg.pos_dyn = 0;
      rg.u_total = a.plan->units_gu;
    }
    __syncthreads();
    sorted = a.sorted_ids;
  }
  cur.n_work = rg.n_work;
  const int u_begin = rg.u_begin, u_end = rg.u_end;
  if (u_begin < u_end) cur.start(rg.w0, rg.ubeg0, rg.pos0);

  const int n_static = u_end - u_begin;
  // The stage has a dynamic tail (kTail instances only: without one the
  // kernel is the plain static split).
  const bool tail = kTail && rg.u_dyn < rg.u_total;
  int* const s_unit = reinterpret_cast<int*>(smem + kStageUnitOff);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    DynTail dt{a.dyn, rg.u_dyn, rg.u_total, 0};
    if (stall_us > 0) return;  // nothing issued, nothing in flight
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int j = 0;
    bool ok = true;
    int tok = 0, tok_i = -1, tok_g = -1;  // lane m: token of member m of the cached group
    // This CTA's static units, then tickets of the dynamic tail until they run
    // out; the first ticket is fetched with the last static unit but one.
    if (tail && n_static == 0) dt.fetch(lane);
    for (;; ++j) {
      int u;
      if (j < n_static) {
        u = u_begin + j;
        if (tail && j == max(n_static - 2, 0)) dt.fetch(lane);
      } else {
        if (!tail) break;
        u = dt.take();
        if (u >= dt.u_total) break;
        if (j == n_static) cur.start(rg.w_dyn, rg.ubeg_dyn, rg.pos_dyn);
        dt.fetch(lane);
      }
      const int s = j % NS, use = j / NS;
      cur.seek(u);
      const int local = u - cur.ubeg;
      const bool tm = cur.tile_major;
      const int grp = tm ? local % cur.groups : local / cur.tiles;
      const int tile = tm ? local / cur.groups : local - grp * cur.tiles;
      const bool shared = cur.expert < 0;
      const int RG = shared ? a.rgs : a.rg;
      const int Iw = shared ? a.Is : a.I;
      const int r0 = tile * RG;
      const int nr = min(RG, Iw - r0);
      const int g0 = grp * xt;
      const int nt = min(xt, cur.n_tok - g0);
      if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
        ok = false;
        break;
      }
      uint8_t* st = stages + (size_t)s * a.stage_bytes;
      const int rb = shared ? d * 2 : rowb;
      const int sb = shared ? 0 : srowb;
      // (int4 boxes always move 8 rows: the byte count says so.)
      const uint32_t bytes = (kFmt && !shared ? (uint32_t)i4g_weight_bytes(d, RG)
                                              : 2u * nr * (rb + sb)) +
                             (uint32_t)nt * d * 2;
      if (lane == 0) {
        if (j >= n_static) s_unit[s] = u;
        mbar_arrive_expect_tx(&full[s], bytes);
      }
      __syncwarp();
      const uint8_t* wbase = shared ? a.sgu : a.gu + (size_t)cur.expert * 2 * a.I * rb;
      // A weight tile that the expert's next token group reads again (the
      // next unit) stays in L2; its last read may go first.
      const uint64_t pol_t = tm && grp + 1 < cur.groups ? pol_x : pol_w;
      int xoff;
      if (kFmt && !shared) {
        // Gate and up codes as one tensor box each (RG rows: I is a multiple
        // of 256, so every unit is whole), their scales as one block each.
        if (lane < 2)
          tma_box_3d(smem_u32(st) + lane * i4g_box_bytes(d, RG), &a.tm_codes, 0,
                     cur.expert * 2 * a.I + lane * Iw + r0, 0, &full[s], pol_t);
        else if (lane < 4) {
          const uint8_t* sbase = reinterpret_cast<const uint8_t*>(a.gu_scales) +
                                 ((size_t)cur.expert * 2 * a.I + (lane - 2) * Iw + r0) * sb;
          bulk_g2s(st + 2 * i4g_box_bytes(d, RG) + (lane - 2) * RG * sb, sbase, RG * sb,
                   &full[s], pol_t);
        }
        xoff = i4g_weight_bytes(d, RG);
      } else {
        if (lane == 0) bulk_g2s(st, wbase + (size_t)r0 * rb, nr * rb, &full[s], pol_t);
        if (lane == 1)
          bulk_g2s(st + RG * rb, wbase + (size_t)(Iw + r0) * rb, nr * rb, &full[s], pol_t);
        xoff = 2 * RG * rb;
      }
      // Token rows of this group (looked up once per (work expert, group)),
      // after the weight copies are under way: they come from L2.  Lane m
      // holds member m's token.
      if (cur.i != tok_i || grp != tok_g) {
        tok_i = cur.i;
        tok_g = grp;
        tok = 0;
        if (lane < nt) {
          tok = g0 + lane;
          if (!shared) {
            const int slot = sorted[cur.pos + g0 + lane];
            tok = slot / a.k;
            if (slot < 0 || tok >= a.T) {
              record_status(a.status, kStatusDeviceCheck);
              tok = 0;
            }
          }
        }
      }
      if (lane < nt)
        bulk_g2s(st + xoff + lane * xp, a.x + (size_t)tok * d, d * 2, &full[s], pol_x);
    }
    if (ok && tail) end_of_units(full, empty, s_unit, j, NS, lane, a.status, ok);
    if (!ok) drain_stages(full, j, NS, a.status);
    return;
  }

  // -------------------------------------------------------------- consumers
  int nred = 0;  // int4 units reduced so far
  for (int j = 0;; ++j) {
    const int s = j % NS, use = j / NS;
    int u;
    if (j < n_static) {
      u = u_begin + j;
    } else {
      // A unit of the dynamic tail, or none: the producer's word in the stage.
      if (!tail) break;
      if (!mbar_wait(&full[s], (uint32_t)(use & 1), a.status, wait_ns)) break;
      u = *reinterpret_cast<volatile int*>(s_unit + s);
      if (u < 0) break;
      if (j == n_static) cur.start(rg.w_dyn, rg.ubeg_dyn, rg.pos_dyn);
    }
    cur.seek(u);
    const int local = u - cur.ubeg;
    const bool tm = cur.tile_major;
    const int grp = tm ? local % cur.groups : local / cur.tiles;
    const int tile = tm ? local / cur.groups : local - grp * cur.tiles;
    const bool shared = cur.expert < 0;
    const int RG = shared ? a.rgs : a.rg;
    const int Iw = shared ? a.Is : a.I;
    const int r0 = tile * RG;
    const int nr = min(RG, Iw - r0);
    const int g0 = grp * xt;
    const int nt = min(xt, cur.n_tok - g0);
    const int rb = shared ? d * 2 : rowb;
    const int sb = shared ? 0 : srowb;
    if (j < n_static && !mbar_wait(&full[s], (uint32_t)(use & 1), a.status, wait_ns)) break;
    const uint32_t st = stages_sa + (uint32_t)(s * a.stage_bytes);
    if (kFmt && !shared) {
      // int4 routed unit on the tensor pipe: RG / 8 tiles of 8 gate + 8 up
      // rows; consumer warp w takes tile tp = w % ntile over the 8-group
      // chunks w / ntile, w / ntile + kConsumerWarps / ntile, ... along d.
      // Warp tp adds the partial sums of the tile's other warps and writes h.
      const int g = lane >> 2, t = lane & 3;
      const int ntile = RG / 8, tp = warp % ntile, r8 = 8 * tp;
      const uint32_t sc = st + 2 * i4g_box_bytes(d, RG);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      gu_int4_mma(st, d, RG, r8, g, t, sc + (r8 + g) * sb, sc + (RG + r8 + g) * sb,
                  st + i4g_weight_bytes(d, RG) + g * xp + 16 * t, g < nt, warp / ntile,
                  kConsumerWarps / ntile, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // Hand-off of the partial sums through one of two buffers, each with a
      // full barrier (the writing warps arrived) and an empty one (the tiles'
      // first warps read).
      const int buf = nred & 1;
      const uint32_t ph = (uint32_t)(nred >> 1) & 1u;
      ++nred;
      float4* red = reinterpret_cast<float4*>(stages + (size_t)NS * a.stage_bytes) +
                    buf * (kConsumerWarps - 1) * 32;
      if (warp >= ntile) {
        if (nred > 2 && !mbar_wait(&red_empty[buf], ph ^ 1u, a.status, wait_ns)) break;
        red[(warp - ntile) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_full[buf]);
        continue;
      }
      if (!mbar_wait(&red_full[buf], ph, a.status, wait_ns)) break;
      for (int w = warp + ntile; w < kConsumerWarps; w += ntile) {
        const float4 o = red[(w - ntile) * 32 + lane];
        acc[0] += o.x;
        acc[1] += o.y;
        acc[2] += o.z;
        acc[3] += o.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[buf]);
      if (r8 + g < nr) {
        // h as two bf16 planes: hi = bf16(h), lo = bf16(h - hi), each row in
        // the down products' k order (i4h_col).
        uint16_t* hh = reinterpret_cast<uint16_t*>(a.h) + (size_t)(cur.pos + g0) * a.I +
                       i4h_col(r0 + r8 + g);
        uint16_t* hl = hh + (size_t)a.h_rows * a.I;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (2 * t + c < nt) {
            const float v = silu(acc[c]) * acc[2 + c];
            const uint16_t hi = bf16_bits(v);
            hh[(size_t)(2 * t + c) * a.I] = hi;
            hl[(size_t)(2 * t + c) * a.I] = bf16_bits(v - __uint_as_float((uint32_t)hi << 16));
          }
        }
      }
      continue;
    }
    // Warp -> (pair p, token subset tsub of nsub): tokens m = tsub + q * nsub.
    const int nsub = kConsumerWarps / RG;
    const int p = warp % RG, tsub = warp / RG;
    const int cnt = (p < nr && nt > tsub) ? (nt - tsub + nsub - 1) / nsub : 0;
    const uint32_t wg = st + p * rb, wu = st + RG * rb + p * rb;
    const uint32_t xs = (uint32_t)(nsub * xp);
    const uint32_t xa = st + 2 * RG * rb + tsub * xp;
    float* hout = shared ? a.hs + (size_t)(g0 + tsub) * a.Is + r0 + p
                         : a.h + (size_t)(cur.pos + g0 + tsub) * a.I + r0 + p;
    const size_t hstride = (size_t)nsub * (shared ? a.Is : a.I);
#define MOE_GU_CASE(N)                                  \
  case N:                                               \
    gu_warp<N>(wg, wu, xa, xs, d, lane, hout, hstride); \
    break;
    switch (cnt) {
      MOE_GU_CASE(1)
      MOE_GU_CASE(2)
      MOE_GU_CASE(3)
      MOE_GU_CASE(4)
      MOE_GU_CASE(5)
      MOE_GU_CASE(6)
      MOE_GU_CASE(7)
      MOE_GU_CASE(8)
      default:
        break;
    }
#undef MOE_GU_CASE
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// --------------------------------------------------------------------------- down
// Consumers: 8 lanes per pair of weight rows, 16 row pairs per pass of the CTA.
template <int kFmt, bool kTail>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    down_kernel(const __grid_constant__ DnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  // int4: the ring starts on a 1024-byte boundary (the swizzled code boxes).
  const uint32_t ring_pad =
      kFmt ? ((1024u - ((smem_u32(smem) + (uint32_t)a.stage_off) & 1023u)) & 1023u) : 0u;
  uint8_t* stages = smem + a.stage_off + ring_pad;
  const uint32_t stages_sa = smem_u32(stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.n_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // The plan does not depend on the gate_up stage: its ids (or the workspace
  // plan) were written by the routing kernels, which completed before the
  // gate_up stage began.  So it is built (or read) before the dependency wait,
  // and the producer then streams the weight rows of its first units, which do
  // not depend on gate_up either; the consumers wait for h.
  const int xt = a.xt;
  const int rowb = kFmt ? a.I / 2 : a.I * 2;
  const int srowb = kFmt ? a.I / 16 : 0;
  UnitCursor cur;
  cur.tiles_r = (int)ceil_div(a.d, a.rd);
  cur.tiles_s = a.Is > 0 ? (int)ceil_div(a.d, a.rds) : 1;
  cur.xt = xt;
  cur.down = true;
  cur.tile_major = kFmt != 0;
  // This CTA's range, in shared memory (read where needed, not held in
  // registers across the unit loops).
  __shared__ CtaRange rg;
  const int32_t* sorted;  // sorted position -> slot (shared or global memory)
  if (a.sp.ids != nullptr) {
    int16_t *wex, *wnt;
    int32_t* ss;
    plan_arrays(smem, a.sp.E, wex, wnt, ss);
    cur.work = nullptr;
    cur.wex = wex;
    cur.wnt = wnt;
    smem_plan(rg, a.sp, a.T, a.k, a.Is > 0, cur.tiles_r, cur.tiles_s, xt, wex, wnt, ss,
                   reinterpret_cast<int*>(stages), a.status);
    sorted = ss;
  } else {
    cur.work = a.work;
    if (threadIdx.x == 0) {
      rg.n_work = a.plan->n_work;
      rg.u_begin = a.cta[blockIdx.x];
      rg.u_end = a.cta[blockIdx.x + 1];
      rg.w0 = a.cta[gridDim.x + 1 + blockIdx.x];
      rg.ubeg0 = rg.pos0 = 0;
      rg.u_dyn = a.cta[gridDim.x];
      rg.w_dyn = a.cta[2 * gridDim.x + 1];
      rg.ubeg_dyn = rg.pos_dyn = 0;
      rg.u_total = a.plan->units_dn;
    }
    __syncthreads();
    sorted = a.sorted_ids;
  }
  cur.n_work = rg.n_work;
  const int u_begin = rg.u_begin, u_end = rg.u_end;
  if (u_begin < u_end) cur.start(rg.w0, rg.ubeg0, rg.pos0);
  if (warp != kConsumerWarps) {
    pdl_wait();
    pdl_trigger();
  }

  const int n_static = u_end - u_begin;
  // The stage has a dynamic tail (kTail instances only: without one the
  // kernel is the plain static split).
  const bool tail = kTail && rg.u_dyn < rg.u_total;
  int* const s_unit = reinterpret_cast<int*>(smem + kStageUnitOff);

  if (warp == kConsumerWarps) {
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_h = policy_evict_last();  // h rows are re-read by every row tile
    DynTail dt{a.dyn, rg.u_dyn, rg.u_total, 0};
    int j = 0;
    bool ok = true;
    const int n_pre = min(NS, n_static);  // units whose weights go before the wait
    for (int pass = 0; pass < 2 && ok; ++pass) {
      // pass 0: weight rows of the first n_pre units; pass 1: everything else:
      // this CTA's static units, then tickets of the dynamic tail until they
      // run out (the first fetched with the last static unit).
      if (pass == 1) {
        pdl_wait();
        pdl_trigger();
        if (blockIdx.x == 0 && lane == 0) *a.dyn_other = 0;
        if (u_begin < u_end) cur.start(rg.w0, rg.ubeg0, rg.pos0);
        if (tail && n_static == 0) dt.fetch(lane);
      }
      for (j = 0;; ++j) {
        int u;
        if (j < n_static) {
          if (pass == 0 && j >= n_pre) break;
          u = u_begin + j;
          if (tail && pass == 1 && j == max(n_static - 2, 0)) dt.fetch(lane);
        } else {
          if (pass == 0 || !tail) break;
          u = dt.take();
          if (u >= dt.u_total) break;
          if (j == n_static) cur.start(rg.w_dyn, rg.ubeg_dyn, rg.pos_dyn);
          dt.fetch(lane);
        }
        const int s = j % NS, use = j / NS;
        cur.seek(u);
        const int local = u - cur.ubeg;
        const bool tm = cur.tile_major;
        const int grp = tm ? local % cur.groups : local / cur.tiles;
        const int tile = tm ? local / cur.groups : local - grp * cur.tiles;
        const bool shared = cur.expert < 0;
        const int RD = shared ? a.rds : a.rd;
        const int Iw = shared ? a.Is : a.I;
        const int r0 = tile * RD;
        const int nr = min(RD, a.d - r0);
        const int g0 = grp * xt;
        const int nt = min(xt, cur.n_tok - g0);
        const bool pre = j < n_pre;  // weights already issued in pass 0
        if (pass == 1 && !pre && use > 0 &&
            !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
          ok = false;
          break;
        }
        uint8_t* st = stages + (size_t)s * a.stage_bytes;
        const int rb = shared ? Iw * 2 : rowb;
        const int sb = shared ? 0 : srowb;
        const bool i4 = kFmt && !shared;
        if (pass == 0 || !pre) {
          // (int4 boxes always move whole 128-row boxes: the byte count says so.)
          const uint32_t bytes = (i4 ? (uint32_t)i4d_codes_bytes(Iw) : (uint32_t)nr * rb) +
                                 (uint32_t)nr * sb + (uint32_t)nt * Iw * 4;
          if (lane == 0) {
            if (j >= n_static) s_unit[s] = u;
            mbar_arrive_expect_tx(&full[s], bytes);
          }
          __syncwarp();
          const uint8_t* wb = shared ? a.sdn : a.dn + (size_t)cur.expert * a.d * rb;
          // A weight tile that the expert's next token group reads again (the
          // next unit) stays in L2; its last read may go first.
          const uint64_t pol_t = tm && grp + 1 < cur.groups ? pol_h : pol_w;
          if (i4) {
            // The code rows as I / 256 swizzled boxes (128 rows each, whatever
            // nr), the scales as one block.
            if (lane < Iw / 256)
              tma_box_2d(smem_u32(st) + lane * kI4DnBox, &a.tm_codes, lane * 128,
                         cur.expert * a.d + r0, &full[s], pol_t);
            if (lane == 31) {
              const uint8_t* sbase =
                  reinterpret_cast<const uint8_t*>(a.dn_scales) + (size_t)cur.expert * a.d * sb;
              bulk_g2s(st + i4d_codes_bytes(Iw), sbase + (size_t)r0 * sb, nr * sb, &full[s],
                       pol_t);
            }
          } else {
            if (lane == 0) bulk_g2s(st, wb + (size_t)r0 * rb, nr * rb, &full[s], pol_t);
          }
        }
        if (pass == 1) {
          if (i4) {
            // The tokens' h rows, both bf16 planes.
            const int hp = i4d_h_pitch(Iw);
            const uint32_t hoff = i4d_codes_bytes(Iw) + RD * sb;
            const uint16_t* h16 = reinterpret_cast<const uint16_t*>(a.h);
            if (lane < 2 * nt) {
              const int m = lane % nt, plane = lane / nt;
              const uint16_t* src =
                  h16 + (size_t)plane * a.h_rows * Iw + (size_t)(cur.pos + g0 + m) * Iw;
              bulk_g2s(st + hoff + (plane * xt + m) * hp, src, Iw * 2, &full[s], pol_h);
            }
          } else if (lane == 2) {
            const float* hsrc =
                shared ? a.hs + (size_t)g0 * Iw : a.h + (size_t)(cur.pos + g0) * Iw;
            bulk_g2s(st + RD * (rb + sb), hsrc, nt * Iw * 4, &full[s], pol_h);
          }
        }
      }
    }
    if (ok && tail) end_of_units(full, empty, s_unit, j, NS, lane, a.status, ok);
    if (!ok) drain_stages(full, j, NS, a.status);
    return;
  }

  const int sub = lane >> 3, sl = lane & 7;  // row within the warp's quad, lane in row
  int slot_of_lane = 0, slot_i = -1, slot_g = -1;  // slot id of token sl of the cached group
  for (int j = 0;; ++j) {
    const int s = j % NS, use = j / NS;
    int u;
    if (j < n_static) {
      u = u_begin + j;
    } else {
      // A unit of the dynamic tail, or none: the producer's word in the stage.
      if (!tail) break;
      if (!mbar_wait(&full[s], (uint32_t)(use & 1), a.status)) break;
      u = *reinterpret_cast<volatile int*>(s_unit + s);
      if (u < 0) break;
      if (j == n_static) cur.start(rg.w_dyn, rg.ubeg_dyn, rg.pos_dyn);
    }
    cur.seek(u);
    const int local = u - cur.ubeg;
    const bool tm = cur.tile_major;
    const int grp = tm ? local % cur.groups : local / cur.tiles;
    const int tile = tm ? local / cur.groups : local - grp * cur.tiles;
    const bool shared = cur.expert < 0;
    const int RD = shared ? a.rds : a.rd;
    const int Iw = shared ? a.Is : a.I;
    const int r0 = tile * RD;
    const int nr = min(RD, a.d - r0);
    const int g0 = grp * xt;
    const int nt = min(xt, cur.n_tok - g0);
    if (cur.i != slot_i || grp != slot_g) {
      slot_i = cur.i;
      slot_g = grp;
      slot_of_lane = (!shared && sl < nt) ? sorted[cur.pos + g0 + sl] : 0;
    }
    const int rb = shared ? Iw * 2 : rowb;
    const int sb = shared ? 0 : srowb;
    if (j < n_static && !mbar_wait(&full[s], (uint32_t)(use & 1), a.status)) break;
    const uint32_t st = stages_sa + (uint32_t)(s * a.stage_bytes);
    if (kFmt && !shared) {
      // int4 routed unit on the tensor pipe: warp w takes rows [16 w, 16 w + 16)
      // of each pass of 16 kConsumerWarps rows.
      const int g = lane >> 2, t = lane & 3;
      const int hp = i4d_h_pitch(Iw);
      const uint32_t sc = st + i4d_codes_bytes(Iw);
      const uint32_t hoff = sc + RD * sb + g * hp + 16 * t;
      const int s0 = 2 * t < nt ? sorted[cur.pos + g0 + 2 * t] : 0;
      const int s1 = 2 * t + 1 < nt ? sorted[cur.pos + g0 + 2 * t + 1] : 0;
      for (int rb0 = warp * 16; rb0 < nr; rb0 += 16 * kConsumerWarps) {
        const int ra = min(rb0 + g, nr - 1), rbb = min(rb0 + g + 8, nr - 1);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        dn_int4_mma(st, ra, rbb, t, sc + ra * sb, sc + rbb * sb, hoff, hoff + xt * hp, g < nt,
                    Iw / 32, acc);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int slot = c ? s1 : s0;
          if (2 * t + c >= nt) continue;
          if (slot < 0 || slot >= a.T * a.k) {
            record_status(a.status, kStatusDeviceCheck);
            continue;
          }
          float* yr = a.y + (size_t)slot * a.d + r0 + rb0;
          if (rb0 + g < nr) yr[g] = acc[c];
          if (rb0 + g + 8 < nr) yr[g + 8] = acc[2 + c];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    const uint32_t ha = st + RD * rb;
    const uint32_t hsb = (uint32_t)Iw * 4u;

    // 8-lane group grp8 (0..15) takes rows grp8 and grp8 + 16 of each 32-row block.
    const int grp8 = warp * 4 + sub;
    for (int rb0 = 0; rb0 < nr; rb0 += 32) {
      const int ra = rb0 + grp8, rbr = rb0 + grp8 + 16;
      const int ca = min(ra, nr - 1), cb = min(rbr, nr - 1);  // clamp: recompute, not written
      const uint32_t wa = st + ca * rb, wb = st + cb * rb;
      float oa = 0.f, ob = 0.f;
#define MOE_DN_CASE(N)                                     \
  case N:                                                  \
    dn_rows2<N>(wa, wb, ha, hsb, Iw, sl, oa, ob);          \
    break;
      switch (nt) {
        MOE_DN_CASE(1)
        MOE_DN_CASE(2)
        MOE_DN_CASE(3)
        MOE_DN_CASE(4)
        MOE_DN_CASE(5)
        MOE_DN_CASE(6)
        MOE_DN_CASE(7)
        MOE_DN_CASE(8)
        default:
          break;
      }
#undef MOE_DN_CASE
      if (sl < nt) {
        if (shared) {
          float* yr = a.ys + (size_t)(g0 + sl) * a.d + r0;
          if (ra < nr) yr[ra] = oa;
          if (rbr < nr) yr[rbr] = ob;
        } else {
          const int slot = slot_of_lane;
          if (slot >= 0 && slot < a.T * a.k) {
            float* yr = a.y + (size_t)slot * a.d + r0;
            if (ra < nr) yr[ra] = oa;
            if (rbr < nr) yr[rbr] = ob;
          } else {
            record_status(a.status, kStatusDeviceCheck);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

}  // namespace

int smem_plan_bytes(int E, int S) {
  return (int)round_up(2 * round_up(2 * (E + 1), 16) + round_up(4 * (int64_t)S, 16), 128);
}

bool smem_plan_fits(const GemvShape& g, int E, int T, int k) {
  return g.n_stages >= 2 && (int64_t)smem_plan_scratch_ints(T * k, E, T) * 4 <=
                                (int64_t)g.n_stages * g.stage_bytes;
}

GemvShape gate_up_shape(int fmt, int d, int I, int Is, int smem_budget, int reserve) {
  (void)I;
  GemvShape g;
  if (fmt) {
    // int4 routed units of 16 gate + 16 up rows (two tensor-pipe tiles), or 8
    // + 8 where d leaves no room for two such stages; shared-expert (bf16)
    // units of up to four row pairs within the routed unit's weight bytes;
    // as many tokens per unit as keep two stages (at most 16 KB of them); the
    // cross-warp partial sums after the ring (and up to 1 KB of alignment).
    const int avail = smem_budget - kBarBytes - reserve - kI4RedBytes - 1024;
    const int xp = x_pitch(1, d);
    int xcap = 16 * 1024 / (d * 2);
    xcap = xcap < 1 ? 1 : (xcap > kMaxXT ? kMaxXT : xcap);
    for (int rg = 16; rg >= 8; rg /= 2) {
      g.rg = rg;
      const int wr = i4g_weight_bytes(d, rg);
      g.rg_shared = kConsumerWarps;
      while (g.rg_shared > 1 && 2 * g.rg_shared * d * 2 > (wr > 16384 ? wr : 16384))
        g.rg_shared /= 2;
      const int w = Is > 0 && 2 * g.rg_shared * d * 2 > wr ? 2 * g.rg_shared * d * 2 : wr;
      g.xt = xcap;
      while (g.xt > 1 && 2 * (int)round_up(w + g.xt * xp, 1024) > avail) --g.xt;
      g.stage_bytes = (int)round_up(w + g.xt * xp, 1024);
      if (2 * g.stage_bytes <= avail) break;
    }
    g.stage_off = kBarBytes + reserve;
    g.n_stages = avail / g.stage_bytes;
    if (g.n_stages > kMaxStages) g.n_stages = kMaxStages;
    return g;
  }
  const int rowr = fmt ? d / 2 + d / 16 : d * 2;
  const int rows = d * 2;
  const int target = 32 * 1024;  // weight bytes per stage
  g.rg = kConsumerWarps;
  while (g.rg > 1 && 2 * g.rg * rowr > target) g.rg /= 2;
  g.rg_shared = kConsumerWarps;
  while (g.rg_shared > 1 && 2 * g.rg_shared * rows > target) g.rg_shared /= 2;
  g.xt = 16 * 1024 / (d * 2);
  g.xt = g.xt < 1 ? 1 : (g.xt > kMaxXT ? kMaxXT : g.xt);
  int w = 2 * g.rg * rowr;
  if (Is > 0 && 2 * g.rg_shared * rows > w) w = 2 * g.rg_shared * rows;
  g.stage_bytes = (int)round_up(w + g.xt * d * 2, 128);
  g.stage_off = kBarBytes + reserve;
  g.n_stages = (smem_budget - g.stage_off) / g.stage_bytes;
  if (g.n_stages > kMaxStages) g.n_stages = kMaxStages;
  return g;
}

GemvShape down_shape(int fmt, int d, int I, int Is, int smem_budget, int reserve) {
  (void)d;
  GemvShape g;
  if (fmt) {
    // int4 routed units: 128 rows (eight m16 tiles, two per consumer warp) as
    // swizzled tensor boxes and the tokens' h rows as two bf16 planes; shared-expert
    // (bf16) units of up to 16 rows within 16 KB with fp32 h rows.
    g.rg = kI4DnRows;
    g.rg_shared = 16;
    while (Is > 0 && g.rg_shared > 4 && g.rg_shared * Is * 2 > 16 * 1024) g.rg_shared /= 2;
    const int imax = Is > I ? Is : I;
    g.xt = 16 * 1024 / (imax * 4);
    g.xt = g.xt < 1 ? 1 : (g.xt > kMaxXT ? kMaxXT : g.xt);
    const int wr = i4d_codes_bytes(I) + g.rg * (I / 16) + 2 * g.xt * i4d_h_pitch(I);
    const int ws = Is > 0 ? g.rg_shared * Is * 2 + g.xt * Is * 4 : 0;
    g.stage_bytes = (int)round_up(wr > ws ? wr : ws, 1024);
    g.stage_off = kBarBytes + reserve;
    g.n_stages = (smem_budget - g.stage_off - 1024) / g.stage_bytes;
    if (g.n_stages > kMaxStages) g.n_stages = kMaxStages;
    return g;
  }
  const int rowr = fmt ? I / 2 + I / 16 : I * 2;
  const int rows = Is * 2;
  const int target = 32 * 1024;
  g.rg = 64;
  while (g.rg > 4 && g.rg * rowr > target) g.rg /= 2;
  g.rg_shared = 64;
  while (Is > 0 && g.rg_shared > 4 && g.rg_shared * rows > target) g.rg_shared /= 2;
  const int imax = Is > I ? Is : I;
  g.xt = 16 * 1024 / (imax * 4);
  g.xt = g.xt < 1 ? 1 : (g.xt > kMaxXT ? kMaxXT : g.xt);
  int w = g.rg * rowr + g.xt * I * 4;
  if (Is > 0 && g.rg_shared * rows + g.xt * Is * 4 > w) w = g.rg_shared * rows + g.xt * Is * 4;
  g.stage_bytes = (int)round_up(w, 128);
  g.stage_off = kBarBytes + reserve;
  g.n_stages = (smem_budget - g.stage_off) / g.stage_bytes;
  if (g.n_stages > kMaxStages) g.n_stages = kMaxStages;
  return g;
}

cudaError_t launch_gate_up(const LaunchCfg& c, const ExpertArgs& e, const GemvShape& g,
                           const uint16_t* x, const int32_t* sorted_ids, const Plan* plan,
                           const WorkExpert* work, const int32_t* cta, const SmemPlanArgs& sp,
                           float* h, float* hs, int* status, int grid, bool tail) {
  GuArgs a;
  memset(&a, 0, sizeof(a));
  if (e.fmt) {
    const uint64_t dims[3] = {128, (uint64_t)e.E * 2 * e.I, (uint64_t)e.d / 256};
    const uint64_t strides[2] = {(uint64_t)e.d / 2, 128};
    const uint32_t box[3] = {128, (uint32_t)g.rg, (uint32_t)e.d / 256};
    if (!encode_map(&a.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, e.gate_up, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  a.sp = sp;
  a.stage_off = g.stage_off;
  a.h_rows = e.h_rows;
  a.cta = cta;
  a.gu = static_cast<const uint8_t*>(e.gate_up);
  a.gu_scales = e.gate_up_scales;
  a.sgu = reinterpret_cast<const uint8_t*>(e.s_gate_up);
  a.sdn = reinterpret_cast<const uint8_t*>(e.s_down);
  a.x = x;
  a.sorted_ids = sorted_ids;
  a.plan = plan;
  a.work = work;
  a.h = h;
  a.hs = hs;
  a.status = status;
  a.dyn = status + kDynCounterBase;
  a.dyn_other = status + kDynCounterBase + 1;
  a.T = e.T;
  a.d = e.d;
  a.I = e.I;
  a.Is = e.Is;
  a.k = e.k;
  a.rg = g.rg;
  a.rgs = g.rg_shared;
  a.xt = g.xt;
  a.stage_bytes = g.stage_bytes;
  a.n_stages = g.n_stages;
  const int smem = g.stage_off + g.stage_bytes * g.n_stages + (e.fmt ? kI4RedBytes + 1024 : 0);
  const void* fn = e.fmt ? (tail ? (const void*)gate_up_kernel<1, true>
                                 : (const void*)gate_up_kernel<1, false>)
                          : (tail ? (const void*)gate_up_kernel<0, true>
                                  : (const void*)gate_up_kernel<0, false>);
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  return launch_kernel(c, fn, dim3(grid), dim3(kThreads), smem, args);
}

cudaError_t launch_down(const LaunchCfg& c, const ExpertArgs& e, const GemvShape& g,
                        const int32_t* sorted_ids, const Plan* plan, const WorkExpert* work,
                        const int32_t* cta, const SmemPlanArgs& sp, const float* h,
                        const float* hs, float* y, float* ys, int* status, int grid, bool tail) {
  DnArgs a;
  memset(&a, 0, sizeof(a));
  if (e.fmt && !encode_map_2d(&a.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, e.down,
                              (uint64_t)e.E * e.d, (uint64_t)e.I / 2, 128, kI4DnRows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.sp = sp;
  a.stage_off = g.stage_off;
  a.h_rows = e.h_rows;
  a.cta = cta;
  a.dn = static_cast<const uint8_t*>(e.down);
  a.dn_scales = e.down_scales;
  a.sdn = reinterpret_cast<const uint8_t*>(e.s_down);
  a.sorted_ids = sorted_ids;
  a.plan = plan;
  a.work = work;
  a.h = h;
  a.hs = hs;
  a.y = y;
  a.ys = ys;
  a.status = status;
  a.dyn = status + kDynCounterBase + 1;
  a.dyn_other = status + kDynCounterBase;
  a.T = e.T;
  a.d = e.d;
  a.I = e.I;
  a.Is = e.Is;
  a.k = e.k;
  a.rd = g.rg;
  a.rds = g.rg_shared;
  a.xt = g.xt;
  a.stage_bytes = g.stage_bytes;
  a.n_stages = g.n_stages;
  const int smem = g.stage_off + g.stage_bytes * g.n_stages + (e.fmt ? 1024 : 0);
  const void* fn = e.fmt ? (tail ? (const void*)down_kernel<1, true>
                                 : (const void*)down_kernel<1, false>)
                          : (tail ? (const void*)down_kernel<0, true>
                                  : (const void*)down_kernel<0, false>);
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  return launch_kernel(c, fn, dim3(grid), dim3(kThreads), smem, args);
}

}  // namespace moe
