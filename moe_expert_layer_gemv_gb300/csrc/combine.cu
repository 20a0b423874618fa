// combine.cu -- weighted top-k combine plus the sigmoid-gated shared expert:
//   out[t] = sum_{j<k} w[t][j] * y[t*k+j] + sigmoid(x[t] . w_sg) * ys[t]
// summed in ascending j, then the shared term, in fp32; rounded to bf16 (RNE).
// No atomics: each output element is produced by one thread, so the result is
// deterministic (the deterministic floor of "Qwen3.8 Flash-Next - GB10
// UltraFast", What this fork adds, removes float atomics from MoE epilogues).
#include <cuda_bf16.h>

#include "launch.h"

namespace moe {

namespace {

constexpr int kThreads = 64;
constexpr int kCols = kThreads * 8;  // output columns per CTA

// grid = (T, ceil(d / kCols)); each thread writes 8 consecutive outputs.
__global__ void __launch_bounds__(kThreads)
    combine_kernel(int d, int k, const float* __restrict__ w, const float* __restrict__ y,
                   const float* __restrict__ ys, const float* __restrict__ sg,
                   const uint16_t* __restrict__ x, const uint16_t* __restrict__ w_sg,
                   uint16_t* __restrict__ out) {
  __shared__ float red[kThreads / 32];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  float gate = 0.f;
  if (ys != nullptr && sg != nullptr) {
    gate = sigmoid(sg[t]);
  } else if (ys != nullptr) {
    // x[t] . w_sg: per-thread strided partials, warp sums, then warps in order.
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const uint4* gr = reinterpret_cast<const uint4*>(w_sg);
    float acc = 0.f;
    for (int c = threadIdx.x; c < d / 8; c += kThreads) {
      const uint4 a = xr[c], b = gr[c];
      acc = fmaf(bf16lo(a.x), bf16lo(b.x), acc);
      acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
      acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc);
      acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
      acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc);
      acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
      acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc);
      acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
    }
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    float z = 0.f;
    for (int q = 0; q < kThreads / 32; ++q) z += red[q];
    gate = sigmoid(z);
  }
  const float* wt = w + (size_t)t * k;
  for (int c = blockIdx.y * kCols + threadIdx.x * 8; c < min(d, (int)(blockIdx.y + 1) * kCols);
       c += kThreads * 8) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    // The shared row and up to eight expert rows are requested before the
    // first product (one round trip to L2 per eight slots), then summed in
    // ascending j and the shared term last.
    float4 sa = make_float4(0.f, 0.f, 0.f, 0.f), sb = sa;
    if (ys != nullptr) {
      const float4* sr = reinterpret_cast<const float4*>(ys + (size_t)t * d + c);
      sa = sr[0];
      sb = sr[1];
    }
    for (int j0 = 0; j0 < k; j0 += 8) {
      float4 ya[8], yb[8];
      float wj[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (j0 + q < k) {
          const float4* yr =
              reinterpret_cast<const float4*>(y + ((size_t)t * k + j0 + q) * d + c);
          ya[q] = yr[0];
          yb[q] = yr[1];
          wj[q] = wt[j0 + q];
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (j0 + q < k) {
          acc[0] = fmaf(wj[q], ya[q].x, acc[0]);
          acc[1] = fmaf(wj[q], ya[q].y, acc[1]);
          acc[2] = fmaf(wj[q], ya[q].z, acc[2]);
          acc[3] = fmaf(wj[q], ya[q].w, acc[3]);
          acc[4] = fmaf(wj[q], yb[q].x, acc[4]);
          acc[5] = fmaf(wj[q], yb[q].y, acc[5]);
          acc[6] = fmaf(wj[q], yb[q].z, acc[6]);
          acc[7] = fmaf(wj[q], yb[q].w, acc[7]);
        }
      }
    }
    if (ys != nullptr) {
      acc[0] = fmaf(gate, sa.x, acc[0]);
      acc[1] = fmaf(gate, sa.y, acc[1]);
      acc[2] = fmaf(gate, sa.z, acc[2]);
      acc[3] = fmaf(gate, sa.w, acc[3]);
      acc[4] = fmaf(gate, sb.x, acc[4]);
      acc[5] = fmaf(gate, sb.y, acc[5]);
      acc[6] = fmaf(gate, sb.z, acc[6]);
      acc[7] = fmaf(gate, sb.w, acc[7]);
    }
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      ow[q] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * d + c) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const LaunchCfg& c, int T, int d, int k, const float* w,
                           const float* y, const float* ys, const float* sg, const uint16_t* x,
                           const uint16_t* w_sg, uint16_t* out) {
  if (T == 0) return cudaSuccess;
  void* args[] = {&d, &k, &w, &y, &ys, &sg, &x, &w_sg, &out};
  return launch_kernel(c, (const void*)combine_kernel, dim3(T, (unsigned)ceil_div(d, kCols)),
                       dim3(kThreads), 0, args);
}

}  // namespace moe
