// expert_gemv.cu -- grouped expert GEMVs for small T (decode / speculative
// verify): gate_up + SwiGLU, then down.  Only the touched experts' weights are
// read, each byte once from HBM ("veloGB10", Kernel work: grouped MoE expert
// kernels that never rebuild full weights; shared-expert work overlapped with
// the MoE step -- here the shared expert is one more work expert in the same
// persistent grid).
//
// Structure (both stages): a persistent grid, one CTA per SM.  Work is cut into
// units = (work expert, token group, row tile); each CTA takes one contiguous
// range of units (its first work expert is precomputed by the plan), so
// consecutive units mostly share an expert and a token group.
// Warp 8 is a producer: one bulk copy (cp.async.bulk, the non-tensor TMA) per
// weight block and per activation row lands a unit in a shared-memory ring
// stage and completes its mbarrier by transaction bytes.  Warps 0-7 consume:
// fp32 dot products out of shared memory, warp-shuffle reductions, the SwiGLU
// (gate_up) or the per-slot output write (down), then release the stage.
// int4 weights are dequantised in registers: (nibble - 8) accumulated against
// the activations per group of 32, times the group's bf16 scale (W4A16 routed
// experts: "Qwen3.8 Flash-Next - GB10 UltraFast", How it works).
#include "launch.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxTokPerWarp = 8;  // gate_up: tokens one warp handles per unit
constexpr int kMaxXT = 8;          // tokens per unit
constexpr int kBarBytes = 256;     // barrier area at the start of shared memory
constexpr int kMaxStages = 8;

struct GuArgs {
  const uint8_t* gu;          // routed gate_up: bf16 [E][2I][d] or codes [E][2I][d/2]
  const uint16_t* gu_scales;  // int4 scales [E][2I][d/32]
  const uint8_t* sgu;         // shared gate_up bf16 [2Is][d] (may be null)
  const uint16_t* x;          // [T][d]
  const int32_t* sorted_ids;
  const Plan* plan;
  const WorkExpert* work;
  const int32_t* cta_first;  // [grid] first work expert of each CTA's range
  float* h;   // [num_post_pad][I]
  float* hs;  // [T][Is]
  int* status;
  int T, d, I, Is, k;
  int rg, rgs, xt, stage_bytes, n_stages;
};

struct DnArgs {
  const uint8_t* dn;          // routed down: bf16 [E][d][I] or codes [E][d][I/2]
  const uint16_t* dn_scales;  // int4 scales [E][d][I/32]
  const uint8_t* sdn;         // shared down bf16 [d][Is]
  const int32_t* sorted_ids;
  const Plan* plan;
  const WorkExpert* work;
  const int32_t* cta_first;
  const float* h;
  const float* hs;
  float* y;   // [T*k][d]
  float* ys;  // [T][d]
  int* status;
  int T, d, I, Is, k;
  int rd, rds, xt, stage_bytes, n_stages;
};

// Walks the work experts along a CTA's contiguous unit range.  Units of one
// work expert are numbered group-major: unit = grp * tiles + tile, so
// consecutive units share a token group (same activation rows).
template <bool kDown>
struct UnitCursor {
  const WorkExpert* work;
  int n_work, tiles_r, tiles_s, xt;
  int i, ubeg, uend, tiles, groups;
  WorkExpert we;
  __device__ __forceinline__ void load(int idx) {
    i = idx;
    we = work[idx];
    tiles = we.expert < 0 ? tiles_s : tiles_r;
    groups = (int)ceil_div(we.n_tok, xt);
    ubeg = kDown ? we.unit_dn : we.unit_gu;
    uend = ubeg + tiles * groups;
  }
  __device__ __forceinline__ void seek(int u) {
    while (u >= uend && i + 1 < n_work) load(i + 1);
  }
};

__device__ __forceinline__ float dot8(uint4 w, uint4 xv, float acc) {
  acc = fmaf(bf16lo(w.x), bf16lo(xv.x), acc);
  acc = fmaf(bf16hi(w.x), bf16hi(xv.x), acc);
  acc = fmaf(bf16lo(w.y), bf16lo(xv.y), acc);
  acc = fmaf(bf16hi(w.y), bf16hi(xv.y), acc);
  acc = fmaf(bf16lo(w.z), bf16lo(xv.z), acc);
  acc = fmaf(bf16hi(w.z), bf16hi(xv.z), acc);
  acc = fmaf(bf16lo(w.w), bf16lo(xv.w), acc);
  acc = fmaf(bf16hi(w.w), bf16hi(xv.w), acc);
  return acc;
}

// Signed int4 value (nibble - 8) as an exact float: (2^23 + nibble) - (2^23 + 8).
__device__ __forceinline__ float nib(uint32_t v, int sh) {
  return __uint_as_float(0x4b000000u | ((v >> sh) & 15u)) - 8388616.0f;
}

// sum_{e<8} (code_e - 8) * x_e for the 8 codes of word v against 8 bf16 of xv.
__device__ __forceinline__ float dot8_int4(uint32_t v, uint4 xv, float acc) {
  acc = fmaf(nib(v, 0), bf16lo(xv.x), acc);
  acc = fmaf(nib(v, 4), bf16hi(xv.x), acc);
  acc = fmaf(nib(v, 8), bf16lo(xv.y), acc);
  acc = fmaf(nib(v, 12), bf16hi(xv.y), acc);
  acc = fmaf(nib(v, 16), bf16lo(xv.z), acc);
  acc = fmaf(nib(v, 20), bf16hi(xv.z), acc);
  acc = fmaf(nib(v, 24), bf16lo(xv.w), acc);
  acc = fmaf(nib(v, 28), bf16hi(xv.w), acc);
  return acc;
}

__device__ __forceinline__ float dot8_f32(uint4 w, float4 a, float4 b, float acc) {
  acc = fmaf(bf16lo(w.x), a.x, acc);
  acc = fmaf(bf16hi(w.x), a.y, acc);
  acc = fmaf(bf16lo(w.y), a.z, acc);
  acc = fmaf(bf16hi(w.y), a.w, acc);
  acc = fmaf(bf16lo(w.z), b.x, acc);
  acc = fmaf(bf16hi(w.z), b.y, acc);
  acc = fmaf(bf16lo(w.w), b.z, acc);
  acc = fmaf(bf16hi(w.w), b.w, acc);
  return acc;
}

__device__ __forceinline__ float dot8_int4_f32(uint32_t v, float4 a, float4 b, float acc) {
  acc = fmaf(nib(v, 0), a.x, acc);
  acc = fmaf(nib(v, 4), a.y, acc);
  acc = fmaf(nib(v, 8), a.z, acc);
  acc = fmaf(nib(v, 12), a.w, acc);
  acc = fmaf(nib(v, 16), b.x, acc);
  acc = fmaf(nib(v, 20), b.y, acc);
  acc = fmaf(nib(v, 24), b.z, acc);
  acc = fmaf(nib(v, 28), b.w, acc);
  return acc;
}

// Producer drain after an abort: wait (bounded) for the last fills of every
// stage so no bulk copy is still writing shared memory when the CTA exits.
__device__ void drain_stages(uint64_t* full, int issued, int n_stages, int* status) {
  for (int j = max(0, issued - n_stages); j < issued; ++j)
    mbar_wait(&full[j % n_stages], (uint32_t)((j / n_stages) & 1), status);
}

// --------------------------------------------------------------------------- gate_up
template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1) gate_up_kernel(const GuArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint8_t* stages = smem + kBarBytes;
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
  pdl_wait();
  pdl_trigger();

  const Plan plan = *a.plan;
  const int d = a.d, nch = d >> 3;
  const int xt = a.xt;
  // Routed row bytes (codes only, for int4) and int4 scale bytes per row.
  const int rowb = kFmt ? d / 2 : d * 2;
  const int srowb = kFmt ? d / 16 : 0;
  const int u_begin = unit_begin(blockIdx.x, plan.units_gu, gridDim.x);
  const int u_end = unit_begin(blockIdx.x + 1, plan.units_gu, gridDim.x);
  UnitCursor<false> cur;
  cur.work = a.work;
  cur.n_work = plan.n_work;
  cur.tiles_r = (int)ceil_div(a.I, a.rg);
  cur.tiles_s = a.Is > 0 ? (int)ceil_div(a.Is, a.rgs) : 1;
  cur.xt = xt;
  if (u_begin < u_end) cur.load(a.cta_first[blockIdx.x]);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int j = 0;
    bool ok = true;
    int tok = 0, tok_i = -1, tok_g = -1;  // lane 4+m: token of member m of the cached group
    for (int u = u_begin; u < u_end; ++u, ++j) {
      const int s = j % NS, use = j / NS;
      cur.seek(u);
      const WorkExpert& we = cur.we;
      const int local = u - cur.ubeg;
      const int grp = local / cur.tiles, tile = local - grp * cur.tiles;
      const bool shared = we.expert < 0;
      const int RG = shared ? a.rgs : a.rg;
      const int Iw = shared ? a.Is : a.I;
      const int r0 = tile * RG;
      const int nr = min(RG, Iw - r0);
      const int g0 = grp * xt;
      const int nt = min(xt, we.n_tok - g0);
      // Token rows of this group: looked up once per (work expert, group).
      if (cur.i != tok_i || grp != tok_g) {
        tok_i = cur.i;
        tok_g = grp;
        tok = 0;
        if (lane >= 4 && lane < 4 + nt) {
          tok = g0 + lane - 4;
          if (!shared) {
            const int slot = a.sorted_ids[we.pos + g0 + lane - 4];
            tok = slot / a.k;
            if (slot < 0 || tok >= a.T) {
              record_status(a.status, kStatusDeviceCheck);
              tok = 0;
            }
          }
        }
      }
      if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
        ok = false;
        break;
      }
      uint8_t* st = stages + (size_t)s * a.stage_bytes;
      const int rb = shared ? d * 2 : rowb;
      const int sb = shared ? 0 : srowb;
      const uint32_t bytes = 2u * nr * (rb + sb) + (uint32_t)nt * d * 2;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
      __syncwarp();
      const uint8_t* wbase = shared ? a.sgu : a.gu + (size_t)we.expert * 2 * a.I * rb;
      if (lane == 0) bulk_g2s(st, wbase + (size_t)r0 * rb, nr * rb, &full[s], pol_w);
      if (lane == 1)
        bulk_g2s(st + RG * rb, wbase + (size_t)(Iw + r0) * rb, nr * rb, &full[s], pol_w);
      if (kFmt && !shared) {
        const uint8_t* sbase =
            reinterpret_cast<const uint8_t*>(a.gu_scales) + (size_t)we.expert * 2 * a.I * sb;
        if (lane == 2)
          bulk_g2s(st + 2 * RG * rb, sbase + (size_t)r0 * sb, nr * sb, &full[s], pol_w);
        if (lane == 3)
          bulk_g2s(st + 2 * RG * rb + RG * sb, sbase + (size_t)(Iw + r0) * sb, nr * sb, &full[s],
                   pol_w);
      }
      const int xoff = 2 * RG * (rb + sb);
      if (lane >= 4 && lane < 4 + nt)
        bulk_g2s(st + xoff + (lane - 4) * d * 2, a.x + (size_t)tok * d, d * 2, &full[s], pol_x);
    }
    if (!ok) drain_stages(full, j, NS, a.status);
    return;
  }

  // -------------------------------------------------------------- consumers
  int j = 0;
  for (int u = u_begin; u < u_end; ++u, ++j) {
    const int s = j % NS, use = j / NS;
    cur.seek(u);
    const WorkExpert& we = cur.we;
    const int local = u - cur.ubeg;
    const int grp = local / cur.tiles, tile = local - grp * cur.tiles;
    const bool shared = we.expert < 0;
    const int RG = shared ? a.rgs : a.rg;
    const int Iw = shared ? a.Is : a.I;
    const int r0 = tile * RG;
    const int nr = min(RG, Iw - r0);
    const int g0 = grp * xt;
    const int nt = min(xt, we.n_tok - g0);
    if (!mbar_wait(&full[s], (uint32_t)(use & 1), a.status)) break;
    const uint8_t* st = stages + (size_t)s * a.stage_bytes;
    const int rb = shared ? d * 2 : rowb;
    const int sb = shared ? 0 : srowb;
    const int p = warp % RG, tsub = warp / RG, nsub = kConsumerWarps / RG;
    const uint4* xs = reinterpret_cast<const uint4*>(st + 2 * RG * (rb + sb));

    if (p < nr) {
      float ag[kMaxTokPerWarp], au[kMaxTokPerWarp];
#pragma unroll
      for (int q = 0; q < kMaxTokPerWarp; ++q) ag[q] = au[q] = 0.f;
      if (kFmt == 0 || shared) {
        const uint4* wg = reinterpret_cast<const uint4*>(st + p * rb);
        const uint4* wu = reinterpret_cast<const uint4*>(st + RG * rb + p * rb);
        for (int c = lane; c < nch; c += 32) {
          const uint4 vg = wg[c], vu = wu[c];
#pragma unroll
          for (int q = 0; q < kMaxTokPerWarp; ++q) {
            const int m = tsub + q * nsub;
            if (m < nt) {
              const uint4 xv = xs[m * nch + c];
              ag[q] = dot8(vg, xv, ag[q]);
              au[q] = dot8(vu, xv, au[q]);
            }
          }
        }
      } else {
        // int4: one 16-byte chunk = 32 codes = one scale group.
        const uint4* cg = reinterpret_cast<const uint4*>(st + p * rb);
        const uint4* cu = reinterpret_cast<const uint4*>(st + RG * rb + p * rb);
        const uint16_t* sg = reinterpret_cast<const uint16_t*>(st + 2 * RG * rb + p * sb);
        const uint16_t* su = reinterpret_cast<const uint16_t*>(st + 2 * RG * rb + RG * sb + p * sb);
        for (int c = lane; c < d / 32; c += 32) {
          const uint4 vg = cg[c], vu = cu[c];
          const float fg = __uint_as_float((uint32_t)sg[c] << 16);
          const float fu = __uint_as_float((uint32_t)su[c] << 16);
#pragma unroll
          for (int q = 0; q < kMaxTokPerWarp; ++q) {
            const int m = tsub + q * nsub;
            if (m < nt) {
              const uint4* xr = xs + m * nch + 4 * c;
              const uint4 x0 = xr[0], x1 = xr[1], x2 = xr[2], x3 = xr[3];
              float pg = dot8_int4(vg.x, x0, 0.f);
              pg = dot8_int4(vg.y, x1, pg);
              pg = dot8_int4(vg.z, x2, pg);
              pg = dot8_int4(vg.w, x3, pg);
              float pu = dot8_int4(vu.x, x0, 0.f);
              pu = dot8_int4(vu.y, x1, pu);
              pu = dot8_int4(vu.z, x2, pu);
              pu = dot8_int4(vu.w, x3, pu);
              ag[q] = fmaf(fg, pg, ag[q]);
              au[q] = fmaf(fu, pu, au[q]);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kMaxTokPerWarp; ++q) {
        const int m = tsub + q * nsub;
        if (m < nt) {
          const float g = warp_sum(ag[q]);
          const float uu = warp_sum(au[q]);
          if (lane == 0) {
            const float hv = silu(g) * uu;
            if (shared)
              a.hs[(size_t)(g0 + m) * a.Is + r0 + p] = hv;
            else
              a.h[(size_t)(we.pos + g0 + m) * a.I + r0 + p] = hv;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// --------------------------------------------------------------------------- down
// Consumers: 8 lanes per weight row, so a warp works on 4 rows at a time.
template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1) down_kernel(const DnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint8_t* stages = smem + kBarBytes;
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
  pdl_wait();
  pdl_trigger();

  const Plan plan = *a.plan;
  const int xt = a.xt;
  const int rowb = kFmt ? a.I / 2 : a.I * 2;
  const int srowb = kFmt ? a.I / 16 : 0;
  const int u_begin = unit_begin(blockIdx.x, plan.units_dn, gridDim.x);
  const int u_end = unit_begin(blockIdx.x + 1, plan.units_dn, gridDim.x);
  UnitCursor<true> cur;
  cur.work = a.work;
  cur.n_work = plan.n_work;
  cur.tiles_r = (int)ceil_div(a.d, a.rd);
  cur.tiles_s = a.Is > 0 ? (int)ceil_div(a.d, a.rds) : 1;
  cur.xt = xt;
  if (u_begin < u_end) cur.load(a.cta_first[blockIdx.x]);

  if (warp == kConsumerWarps) {
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_h = policy_evict_last();  // h rows are re-read by every row tile
    int j = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end; ++u, ++j) {
      const int s = j % NS, use = j / NS;
      cur.seek(u);
      const WorkExpert& we = cur.we;
      const int local = u - cur.ubeg;
      const int grp = local / cur.tiles, tile = local - grp * cur.tiles;
      const bool shared = we.expert < 0;
      const int RD = shared ? a.rds : a.rd;
      const int Iw = shared ? a.Is : a.I;
      const int r0 = tile * RD;
      const int nr = min(RD, a.d - r0);
      const int g0 = grp * xt;
      const int nt = min(xt, we.n_tok - g0);
      if (use > 0 && !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
        ok = false;
        break;
      }
      uint8_t* st = stages + (size_t)s * a.stage_bytes;
      const int rb = shared ? Iw * 2 : rowb;
      const int sb = shared ? 0 : srowb;
      const uint32_t bytes = (uint32_t)nr * (rb + sb) + (uint32_t)nt * Iw * 4;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
      __syncwarp();
      if (lane == 0) {
        const uint8_t* wb = shared ? a.sdn : a.dn + (size_t)we.expert * a.d * rb;
        bulk_g2s(st, wb + (size_t)r0 * rb, nr * rb, &full[s], pol_w);
      }
      if (kFmt && !shared && lane == 1) {
        const uint8_t* sbase =
            reinterpret_cast<const uint8_t*>(a.dn_scales) + (size_t)we.expert * a.d * sb;
        bulk_g2s(st + RD * rb, sbase + (size_t)r0 * sb, nr * sb, &full[s], pol_w);
      }
      if (lane == 2) {
        const float* hsrc = shared ? a.hs + (size_t)g0 * Iw : a.h + (size_t)(we.pos + g0) * Iw;
        bulk_g2s(st + RD * (rb + sb), hsrc, nt * Iw * 4, &full[s], pol_h);
      }
    }
    if (!ok) drain_stages(full, j, NS, a.status);
    return;
  }

  const int sub = lane >> 3, sl = lane & 7;  // row within the warp's quad, lane in row
  int j = 0;
  int slot_of_lane = 0, slot_i = -1, slot_g = -1;  // slot id of token sl of the cached group
  for (int u = u_begin; u < u_end; ++u, ++j) {
    const int s = j % NS, use = j / NS;
    cur.seek(u);
    const WorkExpert& we = cur.we;
    const int local = u - cur.ubeg;
    const int grp = local / cur.tiles, tile = local - grp * cur.tiles;
    const bool shared = we.expert < 0;
    const int RD = shared ? a.rds : a.rd;
    const int Iw = shared ? a.Is : a.I;
    const int r0 = tile * RD;
    const int nr = min(RD, a.d - r0);
    const int g0 = grp * xt;
    const int nt = min(xt, we.n_tok - g0);
    if (cur.i != slot_i || grp != slot_g) {
      slot_i = cur.i;
      slot_g = grp;
      slot_of_lane = (!shared && sl < nt) ? a.sorted_ids[we.pos + g0 + sl] : 0;
    }
    if (!mbar_wait(&full[s], (uint32_t)(use & 1), a.status)) break;
    const uint8_t* st = stages + (size_t)s * a.stage_bytes;
    const int rb = shared ? Iw * 2 : rowb;
    const int sb = shared ? 0 : srowb;
    const float* hsm = reinterpret_cast<const float*>(st + RD * (rb + sb));

    for (int rq = warp * 4; rq < nr; rq += kConsumerWarps * 4) {
      const int r = rq + sub;  // this lane group's row within the tile
      float acc[kMaxXT];
#pragma unroll
      for (int m = 0; m < kMaxXT; ++m) acc[m] = 0.f;
      if (r < nr) {
        if (kFmt == 0 || shared) {
          const uint4* wr = reinterpret_cast<const uint4*>(st + r * rb);
          for (int c = sl; c < Iw / 8; c += 8) {
            const uint4 w = wr[c];
#pragma unroll
            for (int m = 0; m < kMaxXT; ++m) {
              if (m < nt) {
                const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)m * Iw + c * 8);
                acc[m] = dot8_f32(w, hp[0], hp[1], acc[m]);
              }
            }
          }
        } else {
          const uint4* cr = reinterpret_cast<const uint4*>(st + r * rb);
          const uint16_t* sr = reinterpret_cast<const uint16_t*>(st + RD * rb + r * sb);
          for (int c = sl; c < Iw / 32; c += 8) {
            const uint4 v = cr[c];
            const float sc = __uint_as_float((uint32_t)sr[c] << 16);
#pragma unroll
            for (int m = 0; m < kMaxXT; ++m) {
              if (m < nt) {
                const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)m * Iw + c * 32);
                float pp = dot8_int4_f32(v.x, hp[0], hp[1], 0.f);
                pp = dot8_int4_f32(v.y, hp[2], hp[3], pp);
                pp = dot8_int4_f32(v.z, hp[4], hp[5], pp);
                pp = dot8_int4_f32(v.w, hp[6], hp[7], pp);
                acc[m] = fmaf(sc, pp, acc[m]);
              }
            }
          }
        }
      }
      // Reduce across the 8 lanes of each row; lane sl of the group owns token sl.
      float mine = 0.f;
#pragma unroll
      for (int m = 0; m < kMaxXT; ++m) {
        float v = acc[m];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        if (sl == m) mine = v;
      }
      if (r < nr && sl < nt) {
        if (shared) {
          a.ys[(size_t)(g0 + sl) * a.d + r0 + r] = mine;
        } else {
          const int slot = slot_of_lane;
          if (slot >= 0 && slot < a.T * a.k)
            a.y[(size_t)slot * a.d + r0 + r] = mine;
          else
            record_status(a.status, kStatusDeviceCheck);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

}  // namespace

GemvShape gate_up_shape(int fmt, int d, int I, int Is, int smem_budget) {
  (void)I;
  GemvShape g;
  const int rowr = fmt ? d / 2 + d / 16 : d * 2;
  const int rows = d * 2;
  const int target = 32 * 1024;
  g.rg = 8;
  while (g.rg > 1 && 2 * g.rg * rowr > target) g.rg /= 2;
  g.rg_shared = 8;
  while (g.rg_shared > 1 && 2 * g.rg_shared * rows > target) g.rg_shared /= 2;
  g.xt = 16 * 1024 / (d * 2);
  g.xt = g.xt < 1 ? 1 : (g.xt > kMaxXT ? kMaxXT : g.xt);
  int w = 2 * g.rg * rowr;
  if (Is > 0 && 2 * g.rg_shared * rows > w) w = 2 * g.rg_shared * rows;
  g.stage_bytes = (int)round_up(w + g.xt * d * 2, 128);
  g.n_stages = (smem_budget - kBarBytes) / g.stage_bytes;
  if (g.n_stages > kMaxStages) g.n_stages = kMaxStages;
  return g;
}

GemvShape down_shape(int fmt, int d, int I, int Is, int smem_budget) {
  (void)d;
  GemvShape g;
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
  g.n_stages = (smem_budget - kBarBytes) / g.stage_bytes;
  if (g.n_stages > kMaxStages) g.n_stages = kMaxStages;
  return g;
}

cudaError_t launch_gate_up(const LaunchCfg& c, const ExpertArgs& e, const GemvShape& g,
                           const uint16_t* x, const int32_t* sorted_ids, const Plan* plan,
                           const WorkExpert* work, const int32_t* cta_first, float* h, float* hs,
                           int* status, int grid) {
  GuArgs a;
  a.cta_first = cta_first;
  a.gu = static_cast<const uint8_t*>(e.gate_up);
  a.gu_scales = e.gate_up_scales;
  a.sgu = reinterpret_cast<const uint8_t*>(e.s_gate_up);
  a.x = x;
  a.sorted_ids = sorted_ids;
  a.plan = plan;
  a.work = work;
  a.h = h;
  a.hs = hs;
  a.status = status;
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
  const int smem = kBarBytes + g.stage_bytes * g.n_stages;
  const void* fn = e.fmt ? (const void*)gate_up_kernel<1> : (const void*)gate_up_kernel<0>;
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  return launch_kernel(c, fn, dim3(grid), dim3(kThreads), smem, args);
}

cudaError_t launch_down(const LaunchCfg& c, const ExpertArgs& e, const GemvShape& g,
                        const int32_t* sorted_ids, const Plan* plan, const WorkExpert* work,
                        const int32_t* cta_first, const float* h, const float* hs, float* y,
                        float* ys, int* status, int grid) {
  DnArgs a;
  a.cta_first = cta_first;
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
  const int smem = kBarBytes + g.stage_bytes * g.n_stages;
  const void* fn = e.fmt ? (const void*)down_kernel<1> : (const void*)down_kernel<0>;
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  return launch_kernel(c, fn, dim3(grid), dim3(kThreads), smem, args);
}

}  // namespace moe
