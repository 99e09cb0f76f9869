// Activation statistics and activation-aware channel scales.
//
// "AWQ量化实战：无需重训，把大模型压进4bit显存" §2.1: the strength of an input
// channel is the mean of its absolute activations over many calibration
// tokens.  §2.2: salient channels are multiplied by a factor derived from
// that strength; the factor of every channel is a_c^alpha.
#include <mutex>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kColChunks = 32;   // 8-column chunks per block (256 columns)
constexpr int kTokLanes = 8;     // token lanes per block
constexpr int kRun = 16;         // fp32 run length before folding into fp64

int absmean_splits(int64_t T, int K) {
  const int cols_blocks = (K / 8 + kColChunks - 1) / kColChunks;
  int64_t s = (4 * 148 + cols_blocks - 1) / cols_blocks;
  const int64_t max_by_t = (T + 127) / 128;   // at least 128 tokens per split
  if (s > max_by_t) s = max_by_t;
  if (s > 256) s = 256;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

// Partial sums of |x| over one token range for 256 columns; fp32 runs of 16
// tokens are folded into fp64, then the 8 token lanes are added in a fixed
// order.  part[split][col] (fp64).
__global__ void __launch_bounds__(kColChunks* kTokLanes)
    absmean_partial_kernel(const __half* __restrict__ X, int64_t T, int K, int64_t tok_per_split,
                           double* __restrict__ part) {
  __shared__ double red[kTokLanes][kColChunks * 8];
  const int cx = threadIdx.x, ty = threadIdx.y;
  const int col8 = blockIdx.x * kColChunks + cx;   // 8-column chunk index
  const bool valid = col8 * 8 < K;
  const int64_t t0 = blockIdx.y * tok_per_split;
  const int64_t t1 = min(T, t0 + tok_per_split);
  double dacc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) dacc[j] = 0.0;
  if (valid) {
    const __half* base = X + static_cast<size_t>(col8) * 8;
    int64_t t = t0 + ty;
    while (t < t1) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 4
      for (int r = 0; r < kRun && t < t1; ++r, t += kTokLanes) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + static_cast<size_t>(t) * K));
        const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(__habs2(h[j]));
          acc[2 * j] += f.x;
          acc[2 * j + 1] += f.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) dacc[j] += static_cast<double>(acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red[ty][cx * 8 + j] = dacc[j];
  __syncthreads();
  const int tid = ty * kColChunks + cx;   // 0..255 -> one column each
  const int col = blockIdx.x * kColChunks * 8 + tid;
  if (col < K) {
    double s = 0.0;
#pragma unroll
    for (int l = 0; l < kTokLanes; ++l) s += red[l][tid];
    part[static_cast<size_t>(blockIdx.y) * K + col] = s;
  }
}

__global__ void absmean_finalize_kernel(const double* __restrict__ part, int splits, int K,
                                        int64_t T, float* __restrict__ a) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= K) return;
  double s = 0.0;
  for (int i = 0; i < splits; ++i) s += part[static_cast<size_t>(i) * K + c];
  a[c] = static_cast<float>(s / static_cast<double>(T));
}

// s_c = fp32(pow(fp64(max(a, 1e-8f)), alpha)); inv_s = 1 / s_c (IEEE fp32).
__global__ void channel_scales_kernel(const float* __restrict__ a, int K, double alpha,
                                      float* __restrict__ s_c, float* __restrict__ inv_s) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= K) return;
  const float ac = fmaxf(a[c], 1e-8f);
  const float s = static_cast<float>(pow(static_cast<double>(ac), alpha));
  s_c[c] = s;
  inv_s[c] = __fdiv_rn(1.0f, s);
}

}  // namespace

size_t absmean_workspace_size(int64_t T, int K) {
  return static_cast<size_t>(absmean_splits(T, K)) * K * sizeof(double);
}

int launch_absmean(const __half* X, int64_t T, int K, float* a, void* ws, cudaStream_t st) {
  const int splits = absmean_splits(T, K);
  const int64_t per = (T + splits - 1) / splits;
  dim3 grid((K / 8 + kColChunks - 1) / kColChunks, splits);
  dim3 block(kColChunks, kTokLanes);
  double* part = static_cast<double*>(ws);
  absmean_partial_kernel<<<grid, block, 0, st>>>(X, T, K, per, part);
  AWQ_CUDA_TRY_LAUNCH("absmean_partial_kernel");
  absmean_finalize_kernel<<<(K + 255) / 256, 256, 0, st>>>(part, splits, K, T, a);
  AWQ_CUDA_TRY_LAUNCH("absmean_finalize_kernel");
  return AWQ_OK;
}

int launch_channel_scales(const float* a, int K, double alpha, float* s_c, float* inv_s,
                          cudaStream_t st) {
  channel_scales_kernel<<<(K + 255) / 256, 256, 0, st>>>(a, K, alpha, s_c, inv_s);
  AWQ_CUDA_TRY_LAUNCH("channel_scales_kernel");
  return AWQ_OK;
}

}  // namespace awq

// ------------------------------------------------------------------------
// Statistics without any allocation by the caller or the library.
//
// Some callers cannot hand this library device memory at the point of the
// call: runtimes that plan every buffer before execution and forbid
// allocation on the execution path, real-time loops where an allocation's
// latency or possible failure is not acceptable, and plugins whose host
// framework owns all device memory and offers no workspace.  For them the
// partial sums live in a fixed array in this file's device memory (4 MiB,
// held by every GPU that loads the library until the process exits).
namespace awq {
namespace {

constexpr size_t kNoAllocDoubles = (size_t(4) << 20) / sizeof(double);
__device__ __align__(256) double g_absmean_scratch[kNoAllocDoubles];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
double* g_scratch_ptr[kMaxDevices] = {};

// Device address of the fixed array on the current device, looked up once
// per device (the host-side name of the array is not a device address).
int noalloc_scratch(double** out) {
  int dev = 0;
  AWQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("awq_absmean_noalloc: device ordinal %d >= %d is not supported", dev, kMaxDevices);
    return AWQ_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_absmean_scratch);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(g_absmean_scratch)");
    g_scratch_ptr[dev] = static_cast<double*>(p);
  }
  *out = g_scratch_ptr[dev];
  return AWQ_OK;
}

}  // namespace
}  // namespace awq

extern "C" AWQ_API int awq_absmean_noalloc(const uint16_t* X, int64_t T, int32_t K, float* a,
                                           void* stream) {
  using namespace awq;
  if (T <= 0 || K <= 0 || K % kGroup != 0) {
    set_error("awq_absmean_noalloc: T = %lld must be >= 1 and K = %d a positive multiple of 128",
              (long long)T, K);
    return AWQ_ERR_SHAPE;
  }
  if (static_cast<size_t>(K) > kNoAllocDoubles) {
    set_error("awq_absmean_noalloc: K = %d exceeds the fixed scratch limit of %zu input channels",
              K, kNoAllocDoubles);
    return AWQ_ERR_SHAPE;
  }
  if (!X || !a) {
    set_error("awq_absmean_noalloc: X and a must not be NULL");
    return AWQ_ERR_NULL;
  }
  if (!aligned16(X) || !aligned16(a)) {
    set_error("awq_absmean_noalloc: X and a must be 16-byte aligned");
    return AWQ_ERR_ALIGN;
  }
  double* part = nullptr;
  const int rc = noalloc_scratch(&part);
  if (rc != AWQ_OK) return rc;
  int splits = absmean_splits(T, K);
  const int cap = static_cast<int>(kNoAllocDoubles / static_cast<size_t>(K));
  if (splits > cap) splits = cap;
  const int64_t per = (T + splits - 1) / splits;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dim3 grid((K / 8 + kColChunks - 1) / kColChunks, splits);
  dim3 block(kColChunks, kTokLanes);
  // every (split, column) slot that the finalize pass reads is written here,
  // so nothing in the shared array needs clearing between calls
  absmean_partial_kernel<<<grid, block, 0, st>>>(reinterpret_cast<const __half*>(X), T, K, per,
                                                 part);
  AWQ_CUDA_TRY_LAUNCH("absmean_partial_kernel");
  absmean_finalize_kernel<<<(K + 255) / 256, 256, 0, st>>>(part, splits, K, T, a);
  AWQ_CUDA_TRY_LAUNCH("absmean_finalize_kernel");
  return AWQ_OK;
}
