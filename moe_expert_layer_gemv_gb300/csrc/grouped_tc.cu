// grouped_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores for
// prefill-sized T ("veloGB10", Kernel work: grouped MoE expert kernels for
// decode *and prefill*; faster prefill MoE expert kernel and a reworked expert
// schedule).  Two kernels over the moe_align_block_size layout with 128-row
// blocks:
//   gate_up_tc: H[p, n] = silu(X[tok(p)] . Wg[e][n]) * (X[tok(p)] . Wu[e][n])
//   down_tc:    Y[slot(p), :] = H[p] . Wd[e]^T
// where p runs over the padded sorted positions of expert e and tok(p) is the
// token of slot sorted_ids[p] (the shared expert is one more "expert" whose
// rows are the T tokens themselves).
//
// One CTA per SM, persistent, warp-specialised:
//   warp 0      producer: TMA loads into a 4-stage shared-memory ring.  The A
//               tile (128 rows x 64 K) is gathered row by row with
//               cp.async.bulk.tensor ... tile::gather4 (gate_up: rows of x
//               picked through sorted_ids) or loaded tiled (down: rows of H);
//               the B tile (256 weight rows x 64 K) is a tiled load.  Both
//               land 128-byte swizzled, K-major, and complete the stage's
//               mbarrier by transaction bytes.
//   warp 1      one thread issues tcgen05.mma (M=128, N=256, K=16, bf16 in,
//               fp32 accumulate) into one of two TMEM accumulators (2 x 256
//               columns) and releases each stage with tcgen05.commit.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (warp q owns TMEM
//               lanes 32q..32q+31 = tile rows), SwiGLU -> bf16 H (gate_up) or
//               fp32 rows scattered to their slots (down).
// Tiles are (work expert, N block, M block) with the M blocks of one N block
// consecutive, handed to CTAs round-robin, so the CTAs working on an expert's
// weight block at the same time share it through L2.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>

#include "launch.h"

namespace moe {

namespace {

constexpr int kTcThreads = 192;       // 6 warps
constexpr int kTcStages = 4;
constexpr int kTcBM = 128;            // rows per tile (tcgen05 M)
constexpr int kTcBN = 256;            // weight rows per tile (tcgen05 N)
constexpr int kTcBK = 64;             // K per stage: one 128-byte swizzle atom of bf16
constexpr int kTcAStage = kTcBM * kTcBK * 2;  // 16 KB
constexpr int kTcBStage = kTcBN * kTcBK * 2;  // 32 KB
constexpr int kTcStageBytes = kTcAStage + kTcBStage;
constexpr int kTcTmemCols = 2 * kTcBN;  // two accumulators
constexpr int kTcSmemBytes = 1024 + kTcStages * kTcStageBytes + 1024;  // barriers + ring + alignment

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                              ((uint32_t)(kTcBN >> 3) << 17) | ((uint32_t)(kTcBM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: 8-row groups 1024 bytes apart (stride byte offset), the
// leading byte offset unused, descriptor version 1, layout SWIZZLE_128B (2).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kTcIdesc), "r"(accumulate)
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

// Four rows (r0..r3) x one box of columns, landing at 4 consecutive 128-byte rows.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0,
                                            int r1, int r2, int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}

struct TcArgs {
  CUtensorMap tm_a;   // gate_up: x [T][d] box {64, 1} (gather4); down: H [rows][I] box {64, 128}
  CUtensorMap tm_b;   // routed weights: gate_up [E*2I][d] box {64, 128}; down [E*d][I] box {64, 256}
  CUtensorMap tm_bs;  // shared-expert weights, same boxes (unused without a shared expert)
  const int32_t* sorted_ids;
  const Plan* plan;
  const WorkExpert* work;
  uint16_t* h;        // bf16 [rows][I]: routed rows at their sorted positions, shared at hs0 + t
  float* y;           // [T*k][d]
  float* ys;          // [T][d]
  int* status;
  int T, d, I, k, hs0;
  int nb;             // N blocks per expert (gate_up: I / 128; down: d / 256)
  int kb;             // K blocks per tile (gate_up: d / 64; down: I / 64)
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

// kDown = false: gate_up + SwiGLU; true: down.
template <bool kDown>
__global__ void __launch_bounds__(kTcThreads, 1) grouped_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Barriers and the TMEM slot first; the ring starts at the next 1 KB boundary.
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw);
  uint64_t* empty = full + kTcStages;
  uint64_t* acc_full = empty + kTcStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;  // used only after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* n_issued = abort_flag + 1;    // stages filled by the producer
  volatile int* n_consumed = abort_flag + 2;  // stages whose full barrier the MMA thread saw
  const uint32_t ring = (smem_u32(smem_raw) + 1024 + 1023) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = kDown ? 1 : 0;  // WorkExpert pad_ field with the first tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
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
                 "r"(kTcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  const Plan plan = *a.plan;
  const int n_tiles = kDown ? plan.pad_[1] : plan.pad_[0];
  const int S = a.T * a.k;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    int i = 0;
    WorkExpert we = a.work[0];
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      tile_seek(a.work, plan.n_work, slot, t, i, we);
      const bool shared = we.expert < 0;
      const int mblocks = (we.n_tok + kTcBM - 1) / kTcBM;
      const int local = t - we.pad_[slot];
      const int nbk = local / mblocks, mb = local - nbk * mblocks;
      const int row0 = shared ? (kDown ? a.hs0 : 0) + mb * kTcBM : we.pos + mb * kTcBM;
      // gate_up: the tokens of this lane's 4 rows (pads and rows past T read token 0).
      int tok[4] = {0, 0, 0, 0};
      if (!kDown) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int m = mb * kTcBM + lane * 4 + r;  // row within the expert
          if (shared) {
            tok[r] = m < a.T ? m : 0;
          } else if (m < we.n_tok) {
            const int sl = a.sorted_ids[we.pos + m];
            tok[r] = (sl >= 0 && sl < S) ? sl / a.k : 0;
          }
        }
      }
      const CUtensorMap* tb = shared ? &a.tm_bs : &a.tm_b;
      for (int kb = 0; kb < a.kb; ++kb, ++it) {
        const int s = it % kTcStages, use = it / kTcStages;
        if (lane == 0 && use > 0 &&
            !mbar_wait(&empty[s], (uint32_t)((use - 1) & 1), a.status)) {
          *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) {
          ok = false;
          break;
        }
        const uint32_t sa = ring + s * kTcStageBytes, sb = sa + kTcAStage;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], kTcStageBytes);
        __syncwarp();
        const int kx = kb * kTcBK;
        if (kDown) {
          if (lane == 0) tma_load_2d(sa, &a.tm_a, kx, row0, &full[s]);
          if (lane == 1) {
            const int wrow = (shared ? 0 : we.expert * a.d) + nbk * kTcBN;
            tma_load_2d(sb, tb, kx, wrow, &full[s]);
          }
        } else {
          tma_gather4(sa + lane * 4 * 128, &a.tm_a, kx, tok[0], tok[1], tok[2], tok[3], &full[s]);
          if (lane == 0) {
            const int base = shared ? 0 : we.expert * 2 * a.I;
            tma_load_2d(sb, tb, kx, base + nbk * (kTcBN / 2), &full[s]);
            tma_load_2d(sb + kTcBStage / 2, tb, kx, base + a.I + nbk * (kTcBN / 2), &full[s]);
          }
        }
        if (lane == 0) *n_issued = it + 1;
      }
    }
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
        const uint32_t dtm = tmem_base + acc * kTcBN;
        bool ok = true;
        for (int kb = 0; kb < a.kb; ++kb, ++it) {
          const int s = it % kTcStages, use = it / kTcStages;
          if (!mbar_wait(&full[s], (uint32_t)(use & 1), a.status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          *n_consumed = it + 1;
          tc_fence_after();
          const uint32_t sa = ring + s * kTcStageBytes, sb = sa + kTcAStage;
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            umma(dtm, desc_sw128(sa + kk * 32), desc_sw128(sb + kk * 32),
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
    int i = 0;
    WorkExpert we = a.work[0];
    int j = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
      tile_seek(a.work, plan.n_work, slot, t, i, we);
      const bool shared = we.expert < 0;
      const int mblocks = (we.n_tok + kTcBM - 1) / kTcBM;
      const int local = t - we.pad_[slot];
      const int nbk = local / mblocks, mb = local - nbk * mblocks;
      const int acc = j & 1;
      bool ok = true;
      if (lane == 0 && !mbar_wait(&acc_full[acc], (uint32_t)((j >> 1) & 1), a.status)) {
        *abort_flag = 1;
      }
      __syncwarp();
      if (*abort_flag) ok = false;
      if (!ok) break;
      tc_fence_after();
      const int m = mb * kTcBM + q * 32 + lane;  // this thread's row within the expert
      const uint32_t tacc = tmem_base + acc * kTcBN + ((uint32_t)(q * 32) << 16);
      if (!kDown) {
        const int hrow = shared ? a.hs0 + m : we.pos + m;
        uint16_t* hp = a.h + (size_t)hrow * a.I + nbk * (kTcBN / 2);
#pragma unroll 1
        for (int c0 = 0; c0 < kTcBN / 2; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tacc + c0, g);
          tmem_ld32(tacc + kTcBN / 2 + c0, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float h0 = silu(__uint_as_float(g[2 * c])) * __uint_as_float(u[2 * c]);
            const float h1 = silu(__uint_as_float(g[2 * c + 1])) * __uint_as_float(u[2 * c + 1]);
            const __nv_bfloat162 v = __floats2bfloat162_rn(h0, h1);
            packed[c] = *reinterpret_cast<const uint32_t*>(&v);
          }
          uint4* dst = reinterpret_cast<uint4*>(hp + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        }
      } else {
        float* yp = nullptr;
        if (shared) {
          if (m < a.T) yp = a.ys + (size_t)m * a.d + nbk * kTcBN;
        } else if (m < we.n_tok) {
          const int sl = a.sorted_ids[we.pos + m];
          if (sl >= 0 && sl < S) yp = a.y + (size_t)sl * a.d + nbk * kTcBN;
        }
#pragma unroll 1
        for (int c0 = 0; c0 < kTcBN; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tacc + c0, v);
          tmem_ld_wait();
          if (yp != nullptr) {
            uint4* dst = reinterpret_cast<uint4*>(yp + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  // Teardown.  Normally every copy was consumed and every MMA retired before
  // the epilogue saw its last accumulator.  After an abort (a bounded wait ran
  // out), wait -- again bounded -- for the copies still in flight and for the
  // MMAs already issued, so that neither shared memory nor TMEM is written
  // after this CTA releases them.
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int it = *n_consumed; it < *n_issued; ++it)
        mbar_wait(&full[it % kTcStages], (uint32_t)((it / kTcStages) & 1), nullptr);
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
                 "r"(kTcTmemCols)
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
// 128-byte swizzle.
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

}  // namespace

bool tc_supported(int fmt, int d, int I, int Is, int B) {
  return fmt == 0 && B % kTcBM == 0 && I % (kTcBN / 2) == 0 && d % kTcBN == 0 &&
         (Is == 0 || Is == I) && encode_fn() != nullptr;
}

cudaError_t launch_tc(const LaunchCfg& c, bool down, const ExpertArgs& e, const uint16_t* x,
                      const int32_t* sorted_ids, const Plan* plan, const WorkExpert* work,
                      uint16_t* h, int hs0, int h_rows, float* y, float* ys, int* status,
                      int grid) {
  TcArgs a;
  memset(&a, 0, sizeof(a));
  bool ok;
  if (!down) {
    ok = make_map(&a.tm_a, x, (uint64_t)e.T, (uint64_t)e.d, 1) &&
         make_map(&a.tm_b, e.gate_up, (uint64_t)e.E * 2 * e.I, (uint64_t)e.d, kTcBN / 2) &&
         (e.s_gate_up == nullptr ||
          make_map(&a.tm_bs, e.s_gate_up, 2ull * e.Is, (uint64_t)e.d, kTcBN / 2));
    a.nb = e.I / (kTcBN / 2);
    a.kb = e.d / kTcBK;
  } else {
    ok = make_map(&a.tm_a, h, (uint64_t)h_rows, (uint64_t)e.I, kTcBM) &&
         make_map(&a.tm_b, e.down, (uint64_t)e.E * e.d, (uint64_t)e.I, kTcBN) &&
         (e.s_down == nullptr || make_map(&a.tm_bs, e.s_down, (uint64_t)e.d, (uint64_t)e.Is, kTcBN));
    a.nb = e.d / kTcBN;
    a.kb = e.I / kTcBK;
  }
  if (!ok) return cudaErrorInvalidValue;
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
  const void* fn = down ? (const void*)grouped_tc_kernel<true> : (const void*)grouped_tc_kernel<false>;
  cudaError_t err = ensure_smem(fn, kTcSmemBytes);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  return launch_kernel(c, fn, dim3(grid), dim3(kTcThreads), kTcSmemBytes, args);
}

int tc_tiles_per_mblock_gu(int I) { return I / (kTcBN / 2); }
int tc_tiles_per_mblock_dn(int d) { return d / kTcBN; }

}  // namespace moe
