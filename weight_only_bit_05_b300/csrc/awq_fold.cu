// The equivalent transformation folded into the operator that produces the
// quantized layer's input ("什么是激活感知权重量化（AWQ）？", 工作机制):
// out[r][c] = fp16(fp32(W[r][c]) * inv_s[r]), one rounding to nearest.
// HBM-bound elementwise pass: 16-byte loads and stores where the row length
// allows, a grid sized in whole waves of the SMs.
#include "awq_internal.h"

namespace awq {
namespace {

__device__ __forceinline__ __half scale1(__half w, float f) {
  return __float2half_rn(__fmul_rn(__half2float(w), f));
}

// rows whose length is a multiple of 8: one 16-byte vector per step
__global__ void fold_vec8_kernel(const uint4* __restrict__ W, int64_t rows, int64_t cols8,
                                 const float* __restrict__ inv_s, uint4* __restrict__ out) {
  const int64_t n = rows * cols8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float f = __ldg(inv_s + i / cols8);
    uint4 v = W[i];
    __half* h = reinterpret_cast<__half*>(&v);
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = scale1(h[j], f);
    out[i] = v;
  }
}

__global__ void fold_scalar_kernel(const __half* __restrict__ W, int64_t rows, int64_t cols,
                                   const float* __restrict__ inv_s, __half* __restrict__ out) {
  const int64_t n = rows * cols;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = scale1(W[i], __ldg(inv_s + i / cols));
}

}  // namespace

int launch_fold_inv_scales(const __half* W, int64_t rows, int64_t cols, const float* inv_s,
                           __half* out, cudaStream_t st) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  const bool vec = cols % 8 == 0;
  const int64_t items = vec ? rows * (cols / 8) : rows * cols;
  int64_t blocks = (items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;   // 8 CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  if (vec)
    fold_vec8_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
        reinterpret_cast<const uint4*>(W), rows, cols / 8, inv_s, reinterpret_cast<uint4*>(out));
  else
    fold_scalar_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(W, rows, cols, inv_s,
                                                                         out);
  AWQ_CUDA_TRY_LAUNCH(vec ? "fold_vec8_kernel" : "fold_scalar_kernel");
  return AWQ_OK;
}

}  // namespace awq
