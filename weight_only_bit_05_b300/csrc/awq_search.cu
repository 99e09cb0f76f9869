// Activation-aware scale search.
//
// "AWQ量化实战：无需重训，把大模型压进4bit显存" §2.2 (the scale is chosen by a grid
// search so that the quantized layer's output on the calibration tokens
// stays as close as possible to the original), §3.3 第三步/第四步 (collect the
// activation statistics, then search the scale per layer), §5.1 (a single
// coefficient per layer); "什么是激活感知权重量化（AWQ）？" 工作机制 (no
// backpropagation, scales from offline activation statistics).
//
// Flow on one stream, all in this library's kernels:
//   a      = absmean(X_cal)
//   s_c_i  = a^alpha_i, inv_s_i = 1/s_c_i          for all alpha_i at once
//   for each chunk of output rows (Yref kept <= 4 GiB):
//     Yref = X_cal W_chunk^T                        tensor cores, fp32, once
//     for each alpha_i:
//       pack(W_chunk diag(s_c_i))                   bit-exact group RTN
//       X~   = fp16(X_cal * inv_s_i)
//       part = sum over 128 tokens of (X~ W^'^T - Yref)^2 per row (tensor cores)
//       row_err[i][n] = sum of part (fp64, fixed order)
//   mse_i = sum_n row_err[i][n] / (T N)            fp64, fixed order
// The host reads the n_grid errors and takes the first minimum.
#include <vector>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr size_t kYrefBudget = size_t(4) << 30;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct SearchLayout {
  int chunk_rows;
  size_t off_a, off_sc, off_inv, off_stats, off_xt, off_qw, off_sc16, off_zr, off_yref, off_part,
      off_rowerr, off_mse, total;
};

SearchLayout layout(int64_t T, int N, int K, int n_grid) {
  SearchLayout L;
  int64_t rows = static_cast<int64_t>(kYrefBudget / (static_cast<size_t>(T) * 4));
  rows = rows / 128 * 128;
  if (rows < 128) rows = 128;
  const int64_t n_up = (N + 127) / 128 * 128;
  if (rows > n_up) rows = n_up;
  L.chunk_rows = static_cast<int>(rows);
  // packed buffers sized for the largest variant (8-bit codes, 32-channel
  // groups), so that one workspace size serves every configuration
  const int G = K / 32, ZW = (G + 3) / 4;
  size_t o = 0;
  L.off_a = o; o += align256(static_cast<size_t>(K) * 4);
  L.off_sc = o; o += align256(static_cast<size_t>(n_grid) * K * 4);
  L.off_inv = o; o += align256(static_cast<size_t>(n_grid) * K * 4);
  L.off_stats = o; o += align256(absmean_workspace_size(T, K));
  L.off_xt = o; o += align256(static_cast<size_t>(T) * K * 2);
  L.off_qw = o; o += align256(static_cast<size_t>(rows) * K);
  L.off_sc16 = o; o += align256(static_cast<size_t>(rows) * G * 2);
  L.off_zr = o; o += align256(static_cast<size_t>(rows) * ZW * 4);
  L.off_yref = o; o += align256(static_cast<size_t>(T) * rows * 4);
  L.off_part = o; o += align256(static_cast<size_t>(gemm_sqerr_slots(static_cast<int>(T))) * rows * 4);
  L.off_rowerr = o; o += align256(static_cast<size_t>(n_grid) * N * 8);
  L.off_mse = o; o += align256(static_cast<size_t>(n_grid) * 8);
  L.total = o;
  return L;
}

// row_err[r0 + n] = sum over slots of part[slot][n]  (fp64, slot order)
__global__ void rows_reduce_kernel(const float* __restrict__ part, int slots, int ld, int rows,
                                   double* __restrict__ row_err) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= rows) return;
  double s = 0.0;
  for (int i = 0; i < slots; ++i) s += static_cast<double>(part[static_cast<size_t>(i) * ld + n]);
  row_err[n] = s;
}

// mse[i] = sum_n row_err[i][n] / denom, one block per alpha, fixed tree order
__global__ void __launch_bounds__(1024)
    mse_reduce_kernel(const double* __restrict__ row_err, int N, double denom,
                      double* __restrict__ mse) {
  __shared__ double red[1024];
  const double* r = row_err + static_cast<size_t>(blockIdx.x) * N;
  double s = 0.0;
  for (int n = threadIdx.x; n < N; n += blockDim.x) s += r[n];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) mse[blockIdx.x] = red[0] / denom;
}

}  // namespace
}  // namespace awq

using namespace awq;

extern "C" {

size_t awq_search_workspace_size(int64_t T, int32_t N, int32_t K) {
  if (T <= 0 || N <= 0 || K <= 0) return 0;
  return layout(T, N, K, 64).total;
}

int awq_search_scales(const uint16_t* X_cal, int64_t T, const uint16_t* W, int32_t N, int32_t K,
                      const awq_config* cfg, void* workspace, size_t ws_bytes, float* s_c_out,
                      float* inv_s_out, int32_t* best_out, double* mse_out, double* row_err_out,
                      void* stream) {
  NvtxRange range("awq_search_scales");
  const awq_config c = cfg ? *cfg : awq_default_config();
  if ((c.w_bit != 4 && c.w_bit != 8) || (c.group != 128 && c.group != 64 && c.group != 32) ||
      (c.zero_point != 0 && c.zero_point != 1) || c.n_grid < 1 || c.n_grid > 64) {
    set_error("awq_search_scales: unsupported configuration w_bit=%d group=%d zero_point=%d "
              "n_grid=%d", c.w_bit, c.group, c.zero_point, c.n_grid);
    return AWQ_ERR_UNSUPPORTED;
  }
  if (K <= 0 || K % kGroup != 0 || N <= 0 || N % 8 != 0 || T < 1 || T > (int64_t(1) << 30)) {
    set_error("awq_search_scales: bad shape T=%lld N=%d K=%d", (long long)T, N, K);
    return AWQ_ERR_SHAPE;
  }
  const void* ptrs[] = {X_cal, W, s_c_out, inv_s_out};
  const char* names[] = {"X_cal", "W", "s_c_out", "inv_s_out"};
  for (int i = 0; i < 4; ++i) {
    if (!ptrs[i]) {
      set_error("awq_search_scales: %s is NULL", names[i]);
      return AWQ_ERR_NULL;
    }
    if (!aligned16(ptrs[i])) {
      set_error("awq_search_scales: %s is not 16-byte aligned", names[i]);
      return AWQ_ERR_ALIGN;
    }
  }
  if (!best_out || !mse_out) {
    set_error("awq_search_scales: best_out and mse_out (host) are required");
    return AWQ_ERR_NULL;
  }
  if (row_err_out && !aligned16(row_err_out)) {
    set_error("awq_search_scales: row_err_out is not 16-byte aligned");
    return AWQ_ERR_ALIGN;
  }
  const int n_grid = c.n_grid;
  const SearchLayout L = layout(T, N, K, n_grid);
  if (!workspace || !aligned16(workspace) || ws_bytes < awq_search_workspace_size(T, N, K)) {
    set_error("awq_search_scales: workspace must be 16-B aligned and >= %zu bytes",
              awq_search_workspace_size(T, N, K));
    return AWQ_ERR_WORKSPACE;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* a = reinterpret_cast<float*>(ws + L.off_a);
  float* sc_all = reinterpret_cast<float*>(ws + L.off_sc);
  float* inv_all = reinterpret_cast<float*>(ws + L.off_inv);
  __half* xt = reinterpret_cast<__half*>(ws + L.off_xt);
  uint32_t* qw = reinterpret_cast<uint32_t*>(ws + L.off_qw);
  __half* sc16 = reinterpret_cast<__half*>(ws + L.off_sc16);
  uint32_t* zr = reinterpret_cast<uint32_t*>(ws + L.off_zr);
  float* yref = reinterpret_cast<float*>(ws + L.off_yref);
  float* part = reinterpret_cast<float*>(ws + L.off_part);
  double* row_err = reinterpret_cast<double*>(ws + L.off_rowerr);
  double* mse_d = reinterpret_cast<double*>(ws + L.off_mse);
  const __half* X = reinterpret_cast<const __half*>(X_cal);
  const __half* Wh = reinterpret_cast<const __half*>(W);

#define TRY(x)                   \
  do {                           \
    int _s = (x);                \
    if (_s != AWQ_OK) return _s; \
  } while (0)

  TRY(launch_absmean(X, T, K, a, ws + L.off_stats, st));
  for (int i = 0; i < n_grid; ++i)
    TRY(launch_channel_scales(a, K, static_cast<double>(i) / n_grid, sc_all + static_cast<size_t>(i) * K,
                              inv_all + static_cast<size_t>(i) * K, st));
  const int slots = gemm_sqerr_slots(static_cast<int>(T));
  for (int r0 = 0; r0 < N; r0 += L.chunk_rows) {
    const int rows = N - r0 < L.chunk_rows ? N - r0 : L.chunk_rows;
    const __half* Wc = Wh + static_cast<size_t>(r0) * K;
    TRY(launch_gemm(kGemmDenseF32, X, false, static_cast<int>(T), nullptr, nullptr, nullptr, Wc,
                    rows, K, yref, rows, nullptr, 0, st));
    for (int i = 0; i < n_grid; ++i) {
      TRY(launch_pack(Wc, sc_all + static_cast<size_t>(i) * K, rows, K, qw, sc16, zr, st,
                      c.w_bit, c.group, c.zero_point != 0));
      TRY(launch_prescale(X, inv_all + static_cast<size_t>(i) * K, T, K, xt, st, c.w_bit));
      TRY(launch_gemm(kGemmSqErr, xt, true, static_cast<int>(T), qw, sc16, zr, nullptr, rows, K,
                      part, rows, yref, rows, st, c.w_bit, c.group));
      rows_reduce_kernel<<<(rows + 255) / 256, 256, 0, st>>>(
          part, slots, rows, rows, row_err + static_cast<size_t>(i) * N + r0);
      AWQ_CUDA_TRY_LAUNCH("rows_reduce_kernel");
    }
  }
  mse_reduce_kernel<<<n_grid, 1024, 0, st>>>(row_err, N, static_cast<double>(T) * N, mse_d);
  AWQ_CUDA_TRY_LAUNCH("mse_reduce_kernel");
  std::vector<double> mse(n_grid);
  AWQ_CUDA_TRY(cudaMemcpyAsync(mse.data(), mse_d, n_grid * sizeof(double), cudaMemcpyDeviceToHost, st));
  AWQ_CUDA_TRY(cudaStreamSynchronize(st));
  unsigned flags = 0;
  TRY(read_clear_gemm_error(st, &flags));
  if (flags) {
    set_error("awq_search_scales: a tensor-core kernel gave up on a bounded wait (0x%x)", flags);
    return AWQ_ERR_DEVICE;
  }
  int best = 0;
  for (int i = 1; i < n_grid; ++i)
    if (mse[i] < mse[best]) best = i;
  for (int i = 0; i < n_grid; ++i) mse_out[i] = mse[i];
  *best_out = best;
  AWQ_CUDA_TRY(cudaMemcpyAsync(s_c_out, sc_all + static_cast<size_t>(best) * K, K * 4,
                               cudaMemcpyDeviceToDevice, st));
  AWQ_CUDA_TRY(cudaMemcpyAsync(inv_s_out, inv_all + static_cast<size_t>(best) * K, K * 4,
                               cudaMemcpyDeviceToDevice, st));
  if (row_err_out)
    AWQ_CUDA_TRY(cudaMemcpyAsync(row_err_out, row_err, static_cast<size_t>(n_grid) * N * 8,
                                 cudaMemcpyDeviceToDevice, st));
  return AWQ_OK;
#undef TRY
}

}  // extern "C"
