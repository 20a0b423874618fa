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
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
      const float wj = wt[j];
      const float4* yr = reinterpret_cast<const float4*>(y + ((size_t)t * k + j) * d + c);
      const float4 a = yr[0], b = yr[1];
      acc[0] = fmaf(wj, a.x, acc[0]);
      acc[1] = fmaf(wj, a.y, acc[1]);
      acc[2] = fmaf(wj, a.z, acc[2]);
      acc[3] = fmaf(wj, a.w, acc[3]);
      acc[4] = fmaf(wj, b.x, acc[4]);
      acc[5] = fmaf(wj, b.y, acc[5]);
      acc[6] = fmaf(wj, b.z, acc[6]);
      acc[7] = fmaf(wj, b.w, acc[7]);
    }
    if (ys != nullptr) {
      const float4* sr = reinterpret_cast<const float4*>(ys + (size_t)t * d + c);
      const float4 a = sr[0], b = sr[1];
      acc[0] = fmaf(gate, a.x, acc[0]);
      acc[1] = fmaf(gate, a.y, acc[1]);
      acc[2] = fmaf(gate, a.z, acc[2]);
      acc[3] = fmaf(gate, a.w, acc[3]);
      acc[4] = fmaf(gate, b.x, acc[4]);
      acc[5] = fmaf(gate, b.y, acc[5]);
      acc[6] = fmaf(gate, b.z, acc[6]);
      acc[7] = fmaf(gate, b.w, acc[7]);
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
