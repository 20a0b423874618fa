// grouped_tc.cu -- GEMMs on the 5th-generation tensor cores for prefill-sized T
// ("veloGB10", Kernel work: grouped MoE expert kernels for decode *and
// prefill*; faster prefill MoE expert kernel and a reworked expert schedule).
// One persistent, warp-specialised kernel in three modes:
//   gate_up: H[p, n] = silu(X[tok(p)] . Wg[e][n]) * (X[tok(p)] . Wu[e][n])
//   down:    Y[slot(p), :] = H[p] . Wd[e]^T
//   dense:   L[t, e] = X[t] . Wr[e]            (router logits)
// where p runs over the padded sorted positions of expert e (moe_align_block_size
// layout, 128-row blocks) and tok(p) is the token of slot sorted_ids[p]; the
// shared expert is one more "expert" whose rows are the T tokens themselves.
//
// One CTA per SM, 8 warps:
//   warp 0      B producer: weight tiles (BN rows x 64 K, 128-byte swizzled,
//               K-major) by tiled TMA, completing the stage's B barrier by
//               transaction bytes.
//   warps 6-7   A producers: the 128 rows x 64 K activation tile (gate_up: rows
//               of X picked through sorted_ids; down: rows of H; dense: rows of
//               X) with 16-byte cp.async into the same swizzled layout, half the
//               rows each.  A stage's A is published kTcLag stages later, after
//               the warp's copies of it have completed and been fenced for the
//               tensor core.  (A TMA gather moves only 512 bytes per
//               instruction, and one warp issuing both operands stalls each on
//               the other: the memory pipes of the LSU and the TMA unit run in
//               parallel only when different warps feed them.)
//   warp 1      one thread issues tcgen05.mma (M=128, N=BN, K=16, bf16 in, fp32
//               accumulate) into one of two TMEM accumulators and releases each
//               stage with tcgen05.commit.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (warp q owns TMEM lanes
//               32q..32q+31 = tile rows).  gate_up: SwiGLU -> bf16 H rows.
//               down / dense: fp32 rows go through a per-warp shared-memory
//               transpose so that 8 lanes store each 128-byte row segment
//               together (one thread per row would write 16-byte pieces of 32
//               rows per instruction).
// gate_up / down tiles are (work expert, N block, M block) with the M blocks of
// one N block consecutive, handed to CTAs round-robin, so the CTAs working on an
// expert's weight block at the same time share it through L2.  Dense tiles are
// (M block, N block) with the N blocks of one M block consecutive.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>

#include "launch.h"

namespace moe {

namespace {

enum TcMode { kGateUp = 0, kDown = 1, kDense = 2 };

constexpr int kTcBM = 128;                   // rows per tile (tcgen05 M)
constexpr int kTcGatherWarps = 2;            // A producers
constexpr int kTcGatherWarp0 = 6;            // first A producer warp
constexpr int kTcThreads = 32 * (kTcGatherWarp0 + kTcGatherWarps);
constexpr int kTcRowsPerLane = kTcBM / 4 / kTcGatherWarps;  // A rows one lane copies per stage
constexpr int kTcBK = 64;                    // K per stage: one 128-byte swizzle atom of bf16
constexpr int kTcAStage = kTcBM * kTcBK * 2;  // 16 KB
constexpr int kTcRingBytes = 192 * 1024;     // stage ring
constexpr int kTcLag = 2;                    // gathered stages in flight before publication
constexpr int kTcStgStride = 36;             // floats per row of the epilogue transpose
constexpr int kTcStgBytes = 4 * 32 * kTcStgStride * 4;
constexpr int kTcHeadBytes = 1024;           // barriers, TMEM slot, flags

template <int BN>
struct TcCfg {
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "N tile");
  static constexpr int kBStage = BN * kTcBK * 2;
  static constexpr int kStageBytes = kTcAStage + kBStage;
  static constexpr int kStages = kTcRingBytes / kStageBytes > 8 ? 8 : kTcRingBytes / kStageBytes;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators (a power of two >= 32)
  static constexpr int kSmemBytes = kTcHeadBytes + kStages * kStageBytes + 1024 + kTcStgBytes;
  // Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
  // N >> 3 at bit 17, M >> 4 at bit 24.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     ((uint32_t)(BN >> 3) << 17) |
                                     ((uint32_t)(kTcBM >> 4) << 24);
};
static_assert(TcCfg<256>::kStages > kTcLag, "the gather lag must leave stages to consume");
static_assert(TcCfg<256>::kSmemBytes <= 227 * 1024, "shared memory");

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: 8-row groups 1024 bytes apart (stride byte offset), the
// leading byte offset unused, descriptor version 1, layout SWIZZLE_128B (2).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte global -> shared copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Orders this thread's completed shared-memory writes before later reads of
// the same bytes by the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct TcArgs {
  CUtensorMap tm_b;   // gate_up [E*2I][d] box {64, BN/2}; down [E*d][I] / dense [E][d] box {64, BN}
  CUtensorMap tm_bs;  // shared-expert weights, same boxes (unused without a shared expert)
  const uint16_t* x;  // X [T][d] (gate_up, dense)
  const int32_t* sorted_ids;
  const Plan* plan;
  const WorkExpert* work;
  uint16_t* h;        // bf16 [h_rows][I]: routed rows at their sorted positions, shared at hs0 + t
  float* y;           // down: [T*k][d]; dense: logits [T][ld_out]
  float* ys;          // down: [T][d]
  int* status;
  int T, d, I, k, hs0;
  int nb;             // N blocks per expert (gate_up: I / (BN/2); down: d / BN; dense: E / BN)
  int kb;             // K blocks per tile (gate_up, dense: d / 64; down: I / 64)
  int dense_tiles;    // dense: ceil(T / 128) * nb
  int ld_out;         // dense: row stride of the logits
};

// Which work expert holds tile t (tiles numbered per the plan, WorkExpert
// field pad_[slot] = first tile); cursor i only moves forward.
__device__ __forceinline__ void tile_seek(const WorkExpert* work, int n_work, int slot, int t,
                                          int& i, WorkExpert& we) {
  while (i + 1 < n_work && work[i + 1].pad_[slot] <= t) {
    ++i;
    we = work[i];
  }
}

// Tile t of a grouped mode: expert record, N block, M block.
struct TileIdx {
  bool shared;
  int nbk, mb;
};
__device__ __forceinline__ TileIdx grouped_tile(const WorkExpert& we, int slot, int t) {
  TileIdx ti;
  ti.shared = we.expert < 0;
  const int mblocks = (we.n_tok + kTcBM - 1) / kTcBM;
  const int local = t - we.pad_[slot];
  ti.nbk = local / mblocks;
  ti.mb = local - ti.nbk * mblocks;
  return ti;
}

// silu(g) * u with the fast exponential and division intrinsics (a few ulp of
// fp32; the result is rounded to bf16).  For g -> -inf the divisor overflows
// and the quotient is 0, the limit of silu.
__device__ __forceinline__ float swiglu_fast(float g, float u) {
  return __fdividef(g * u, 1.0f + __expf(-g));
}

// fp32 epilogue of one accumulator (down / dense): row `lane` of this warp's
// 32 rows goes to rowp (nullptr = not stored), columns [0, BN).  Each 32-column
// slice passes through the warp's transpose buffer so that stores are 128-byte
// row segments.
template <int BN>
__device__ __forceinline__ void store_rows_f32(uint32_t tacc, float* rowp, float* stg, int lane) {
  const unsigned long long mine = reinterpret_cast<unsigned long long>(rowp);
  const int sub = lane >> 3, ch = lane & 7;
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tacc + c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(stg + lane * kTcStgStride + 4 * j) =
          make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int r = 4 * p + sub;
      float* dst = reinterpret_cast<float*>(__shfl_sync(0xffffffffu, mine, r));
      const uint4 val = *reinterpret_cast<const uint4*>(stg + r * kTcStgStride + 4 * ch);
      if (dst != nullptr) *reinterpret_cast<uint4*>(dst + c0 + 4 * ch) = val;
    }
    __syncwarp();
  }
}

template <int kMode, int BN>
__global__ void __launch_bounds__(kTcThreads, 1) grouped_tc_kernel(const __grid_constant__ TcArgs a) {
  using Cfg = TcCfg<BN>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Head (barriers, TMEM slot, flags), then the ring at the next 1 KB boundary,
  // then the epilogue transpose buffers.
  uint64_t* full_b = reinterpret_cast<uint64_t*>(smem_raw);  // B landed (transaction bytes)
  uint64_t* full_a = full_b + NS;                             // A published by every A producer
  uint64_t* empty = full_a + NS;
  uint64_t* acc_full = empty + NS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;  // used only after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* n_issued = abort_flag + 1;    // stages whose B copy warp 0 issued
  volatile int* n_consumed = abort_flag + 2;  // stages whose barriers the MMA thread saw
  const uint32_t ring = (smem_u32(smem_raw) + kTcHeadBytes + 1023) & ~1023u;
  float* stg_all = reinterpret_cast<float*>(smem_raw + (ring - smem_u32(smem_raw)) +
                                            NS * Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = kMode == kDown ? 1 : 0;  // WorkExpert pad_ field with the first tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&full_a[s], kTcGatherWarps);
      mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&acc_full[c], 1);
      mbar_init(&acc_empty[c], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *n_issued = 0;
    *n_consumed = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(Cfg::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  Plan plan;
  int n_tiles;
  if (kMode == kDense) {
    plan.n_work = 0;
    n_tiles = a.dense_tiles;
  } else {
    plan = *a.plan;
    n_tiles = kMode == kDown ? plan.pad_[1] : plan.pad_[0];
  }
  const int S = a.T * a.k;

  if (warp == 0) {
    // ------------------------------------------------------------ B producer
    int i = 0;
    WorkExpert we;
    if (kMode != kDense) we = a.work[0];
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      TileIdx ti;
      if (kMode == kDense) {
        ti.shared = false;
        ti.mb = t / a.nb;
        ti.nbk = t - ti.mb * a.nb;
      } else {
        tile_seek(a.work, plan.n_work, slot, t, i, we);
        ti = grouped_tile(we, slot, t);
      }
      const CUtensorMap* tb = ti.shared ? &a.tm_bs : &a.tm_b;
      for (int kb = 0; kb < a.kb; ++kb, ++it) {
        const int s = it % NS, use = it / NS;
        if (lane == 0 && use > 0 &&
            !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
          *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sb = ring + s * Cfg::kStageBytes + kTcAStage;
          const int kx = kb * kTcBK;
          mbar_arrive_expect_tx(&full_b[s], Cfg::kBStage);
          if (kMode == kGateUp) {
            const int base = ti.shared ? 0 : we.expert * 2 * a.I;
            tma_load_2d(sb, tb, kx, base + ti.nbk * (BN / 2), &full_b[s]);
            tma_load_2d(sb + Cfg::kBStage / 2, tb, kx, base + a.I + ti.nbk * (BN / 2), &full_b[s]);
          } else if (kMode == kDown) {
            tma_load_2d(sb, tb, kx, (ti.shared ? 0 : we.expert * a.d) + ti.nbk * BN, &full_b[s]);
          } else {
            tma_load_2d(sb, tb, kx, ti.nbk * BN, &full_b[s]);
          }
          *n_issued = it + 1;
        }
      }
    }
  } else if (warp >= kTcGatherWarp0) {
    // ------------------------------------------------------------ A producers
    const int g = warp - kTcGatherWarp0;
    const int sub = lane >> 3, ch = lane & 7;  // rows 4 j + sub, 16-byte chunk ch
    const uint16_t* asrc = kMode == kDown ? a.h : a.x;
    int i = 0;
    WorkExpert we;
    if (kMode != kDense) we = a.work[0];
    int it = 0, published = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      TileIdx ti;
      if (kMode == kDense) {
        ti.shared = false;
        ti.mb = t / a.nb;
        ti.nbk = t - ti.mb * a.nb;
      } else {
        tile_seek(a.work, plan.n_work, slot, t, i, we);
        ti = grouped_tile(we, slot, t);
      }
      // Element offsets of this lane's source rows (-1: a pad row, zero-filled).
      int roff[kTcRowsPerLane];
#pragma unroll
      for (int jj = 0; jj < kTcRowsPerLane; ++jj) {
        const int m = ti.mb * kTcBM + 4 * (g * kTcRowsPerLane + jj) + sub;  // row within the expert
        int o = -1;
        if (kMode == kDown) {
          o = ((ti.shared ? a.hs0 : we.pos) + m) * a.I;
        } else if (kMode == kDense || ti.shared) {
          if (m < a.T) o = m * a.d;
        } else if (m < we.n_tok) {
          const int sl = a.sorted_ids[we.pos + m];
          if (sl >= 0 && sl < S) o = (sl / a.k) * a.d;
        }
        roff[jj] = o;
      }
      for (int kb = 0; kb < a.kb; ++kb, ++it) {
        const int s = it % NS, use = it / NS;
        if (lane == 0 && use > 0 &&
            !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
          *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) {
          ok = false;
          break;
        }
        const uint32_t sa = ring + s * Cfg::kStageBytes;
        const int kx = kb * kTcBK;
        // Row r of the tile lands at r * 128 with its 16-byte chunks permuted by
        // r mod 8: the layout a 128-byte-swizzled TMA box would produce.
#pragma unroll
        for (int jj = 0; jj < kTcRowsPerLane; ++jj) {
          const int r = 4 * (g * kTcRowsPerLane + jj) + sub;
          const uint32_t dst = sa + r * 128 + ((ch ^ (r & 7)) << 4);
          const uint16_t* src = asrc + (roff[jj] < 0 ? 0 : roff[jj] + kx + 8 * ch);
          cp_async16(dst, src, roff[jj] < 0 ? 0u : 16u);
        }
        cp_async_commit();
        if (it + 1 - published > kTcLag) {
          cp_async_wait<kTcLag>();
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full_a[published % NS]);
          ++published;
        }
      }
    }
    // Publish the stages still held back (also after an abort: the MMA thread
    // may be waiting for them; every copy of this warp has landed by now).
    cp_async_wait<0>();
    fence_proxy_async();
    __syncwarp();
    if (lane == 0)
      for (; published < it; ++published) mbar_arrive(&full_a[published % NS]);
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, j = 0;
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
        const int acc = j & 1;
        if (j >= 2 && !mbar_wait(&acc_empty[acc], (uint32_t)(((j >> 1) - 1) & 1), a.status)) {
          *abort_flag = 1;
        }
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t dtm = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < a.kb; ++kb, ++it) {
          const int s = it % NS, use = it / NS;
          if (!mbar_wait(&full_b[s], (uint32_t)(use & 1), a.status) ||
              !mbar_wait(&full_a[s], (uint32_t)(use & 1), a.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          *n_consumed = it + 1;
          tc_fence_after();
          const uint32_t sa = ring + s * Cfg::kStageBytes, sb = sa + kTcAStage;
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            umma(dtm, desc_sw128(sa + kk * 32), desc_sw128(sb + kk * 32), Cfg::kIdesc,
                 (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);  // accumulator ready for the epilogue
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    float* stg = stg_all + q * 32 * kTcStgStride;
    int i = 0;
    WorkExpert we;
    if (kMode != kDense) we = a.work[0];
    int j = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
      TileIdx ti;
      if (kMode == kDense) {
        ti.shared = false;
        ti.mb = t / a.nb;
        ti.nbk = t - ti.mb * a.nb;
      } else {
        tile_seek(a.work, plan.n_work, slot, t, i, we);
        ti = grouped_tile(we, slot, t);
      }
      const int acc = j & 1;
      if (lane == 0 && !mbar_wait(&acc_full[acc], (uint32_t)((j >> 1) & 1), a.status)) {
        *abort_flag = 1;
      }
      __syncwarp();
      if (*abort_flag) break;
      tc_fence_after();
      const int m = ti.mb * kTcBM + q * 32 + lane;  // this thread's row within the expert
      const uint32_t tacc = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      if (kMode == kGateUp) {
        const int hrow = ti.shared ? a.hs0 + m : we.pos + m;
        uint16_t* hp = a.h + (size_t)hrow * a.I + ti.nbk * (BN / 2);
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tacc + c0, g);
          tmem_ld32(tacc + BN / 2 + c0, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float h0 = swiglu_fast(__uint_as_float(g[2 * c]), __uint_as_float(u[2 * c]));
            const float h1 =
                swiglu_fast(__uint_as_float(g[2 * c + 1]), __uint_as_float(u[2 * c + 1]));
            const __nv_bfloat162 v = __floats2bfloat162_rn(h0, h1);
            packed[c] = *reinterpret_cast<const uint32_t*>(&v);
          }
          uint4* dst = reinterpret_cast<uint4*>(hp + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        }
      } else {
        float* rowp = nullptr;
        if (kMode == kDense) {
          if (m < a.T) rowp = a.y + (size_t)m * a.ld_out + ti.nbk * BN;
        } else if (ti.shared) {
          if (m < a.T) rowp = a.ys + (size_t)m * a.d + ti.nbk * BN;
        } else if (m < we.n_tok) {
          const int sl = a.sorted_ids[we.pos + m];
          if (sl >= 0 && sl < S) rowp = a.y + (size_t)sl * a.d + ti.nbk * BN;
        }
        store_rows_f32<BN>(tacc, rowp, stg, lane);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  // Teardown.  Normally every copy was consumed and every MMA retired before
  // the epilogue saw its last accumulator.  After an abort (a bounded wait ran
  // out), wait -- again bounded -- for the B copies still in flight (the A
  // producers drained their own copies above) and for the MMAs already issued,
  // so that neither shared memory nor TMEM is written after this CTA releases
  // them.
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int it = *n_consumed; it < *n_issued; ++it)
        mbar_wait(&full_b[it % NS], (uint32_t)((it / NS) & 1), nullptr);
    }
    if (warp == 1 && lane == 0) {
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(Cfg::kTmemCols)
                 : "memory");
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D bf16 tensor map over [rows][cols] (row-major), box {64 cols, box_rows},
// 128-byte swizzle; reads past the last row return zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kTcBNExpert = 256;  // N tile of the expert GEMMs
constexpr int kTcBNRouter = 64;   // N tile of the router GEMM (E / 64 tiles per M block)

template <int kMode, int BN>
cudaError_t launch_mode(const LaunchCfg& c, TcArgs& a, int grid) {
  const void* fn = (const void*)grouped_tc_kernel<kMode, BN>;
  cudaError_t err = ensure_smem(fn, TcCfg<BN>::kSmemBytes);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  return launch_kernel(c, fn, dim3(grid), dim3(kTcThreads), TcCfg<BN>::kSmemBytes, args);
}

}  // namespace

bool tc_supported(int fmt, int d, int I, int Is, int B) {
  return fmt == 0 && B % kTcBM == 0 && I % (kTcBNExpert / 2) == 0 && d % kTcBNExpert == 0 &&
         (Is == 0 || Is == I) && encode_fn() != nullptr;
}

bool tc_router_supported(int T, int d, int E) {
  return E % kTcBNRouter == 0 && d % kTcBK == 0 && (int64_t)T * d < (1ll << 31) &&
         encode_fn() != nullptr;
}

cudaError_t launch_tc(const LaunchCfg& c, bool down, const ExpertArgs& e, const uint16_t* x,
                      const int32_t* sorted_ids, const Plan* plan, const WorkExpert* work,
                      uint16_t* h, int hs0, int h_rows, float* y, float* ys, int* status,
                      int grid) {
  constexpr int BN = kTcBNExpert;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  bool ok;
  if (!down) {
    if ((int64_t)e.T * e.d >= (1ll << 31)) return cudaErrorInvalidValue;
    ok = make_map(&a.tm_b, e.gate_up, (uint64_t)e.E * 2 * e.I, (uint64_t)e.d, BN / 2) &&
         (e.s_gate_up == nullptr ||
          make_map(&a.tm_bs, e.s_gate_up, 2ull * e.Is, (uint64_t)e.d, BN / 2));
    a.nb = e.I / (BN / 2);
    a.kb = e.d / kTcBK;
  } else {
    if ((int64_t)h_rows * e.I >= (1ll << 31)) return cudaErrorInvalidValue;
    ok = make_map(&a.tm_b, e.down, (uint64_t)e.E * e.d, (uint64_t)e.I, BN) &&
         (e.s_down == nullptr || make_map(&a.tm_bs, e.s_down, (uint64_t)e.d, (uint64_t)e.Is, BN));
    a.nb = e.d / BN;
    a.kb = e.I / kTcBK;
  }
  if (!ok) return cudaErrorInvalidValue;
  a.x = x;
  a.sorted_ids = sorted_ids;
  a.plan = plan;
  a.work = work;
  a.h = h;
  a.y = y;
  a.ys = ys;
  a.status = status;
  a.T = e.T;
  a.d = e.d;
  a.I = e.I;
  a.k = e.k;
  a.hs0 = hs0;
  return down ? launch_mode<kDown, BN>(c, a, grid) : launch_mode<kGateUp, BN>(c, a, grid);
}

cudaError_t launch_tc_router(const LaunchCfg& c, const uint16_t* x, const uint16_t* wr,
                             float* logits, int T, int d, int E, int* status, int sms) {
  constexpr int BN = kTcBNRouter;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_map(&a.tm_b, wr, (uint64_t)E, (uint64_t)d, BN)) return cudaErrorInvalidValue;
  a.x = x;
  a.y = logits;
  a.status = status;
  a.T = T;
  a.d = d;
  a.k = 1;
  a.nb = E / BN;
  a.kb = d / kTcBK;
  a.dense_tiles = (int)ceil_div(T, kTcBM) * a.nb;
  a.ld_out = E;
  const int grid = a.dense_tiles < sms ? a.dense_tiles : sms;
  return launch_mode<kDense, BN>(c, a, grid);
}

int tc_tiles_per_mblock_gu(int I) { return I / (kTcBNExpert / 2); }
int tc_tiles_per_mblock_dn(int d) { return d / kTcBNExpert; }

}  // namespace moe
